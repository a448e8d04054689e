"""Pins for oracle.attention: brute force, Eqs. 22/24/26, split-K combine."""
import math

import numpy as np
import pytest

from oracle import attention, cache, quant, rotations


def _brute_decode(q, k_hat, v_hat, r_k, gqa):
    """Pure-Python loops: q' = q R, a_s = q'.k_s / sqrt(d), softmax, o = sum p v."""
    hq = len(q)
    n = len(k_hat)
    out = []
    for j in range(hq):
        h = j // gqa
        qr = [sum(q[j][c] * r_k[h][c][d] for c in range(128)) for d in range(128)]
        a = [sum(qr[d] * k_hat[s][h][d] for d in range(128)) / math.sqrt(128) for s in range(n)]
        m = max(a)
        e = [math.exp(x - m) for x in a]
        z = sum(e)
        out.append([sum(e[s] / z * v_hat[s][h][d] for s in range(n)) for d in range(128)])
    return np.array(out)


def test_decode_attention_matches_brute_force_loops():
    g = np.random.default_rng(0)
    hq, hkv, n = 4, 2, 6
    q = g.standard_normal((hq, 128))
    kh = g.standard_normal((n, hkv, 128)) * 2
    vh = g.standard_normal((n, hkv, 128))
    rk = np.stack([rotations.expm_skew(g.normal(0, 0.1, (128, 128))) for _ in range(hkv)])
    got = attention.decode_attention(q, kh, vh, rk, 2)
    ref = _brute_decode(q.tolist(), kh.tolist(), vh.tolist(), rk.tolist(), 2)
    assert np.abs(got - ref).max() < 1e-12


def test_rotated_query_equals_inverse_rotated_key():
    # Eqs. 22/26: q (k_R R^T)^T = (q R) k_R^T
    g = np.random.default_rng(1)
    r = rotations.expm_skew(g.normal(0, 0.05, (128, 128)))
    q = g.standard_normal(128)
    k_r = quant.quant_dequant(g.standard_normal((10, 128)) @ r, 1.0)
    assert np.abs(q @ (k_r @ r.T).T - (q @ r) @ k_r.T).max() < 1e-12


def test_key_centring_leaves_softmax_unchanged():
    # Eq. 24: (q R)((k - mu) R)^T = q (k - mu)^T = q k^T - q mu^T, constant in s
    g = np.random.default_rng(2)
    k = g.standard_normal((50, 128)) + 10 * (g.random(128) < 0.05)
    mu = k.mean(axis=0)
    q = g.standard_normal(128)
    r = rotations.signed_hadamard(np.where(g.random(128) < .5, -1., 1.))
    a = k @ q / np.sqrt(128)
    a_c = ((k - mu) @ r) @ (q @ r) / np.sqrt(128)
    assert np.abs((a - a_c) - (q @ mu) / np.sqrt(128)).max() < 1e-11
    assert np.abs(attention.softmax(a) - attention.softmax(a_c)).max() < 1e-12


@pytest.mark.parametrize("n_splits", [1, 2, 3, 7, 64])
def test_split_k_equals_unsplit(n_splits):
    g = np.random.default_rng(3)
    hq, hkv, n = 8, 2, 301
    q = g.standard_normal((hq, 128)) * 3
    kh = g.standard_normal((n, hkv, 128))
    vh = g.standard_normal((n, hkv, 128))
    rk = np.stack([np.eye(128)] * hkv)
    a = attention.decode_attention(q, kh, vh, rk, 4)
    b = attention.split_decode_attention(q, kh, vh, rk, 4, n_splits)
    assert np.abs(a - b).max() < 1e-12


def test_gqa_head_mapping():
    # query head j reads KV head j // g: make KV heads distinguishable by their values
    n, hkv, g_ = 5, 3, 2
    kh = np.zeros((n, hkv, 128))
    vh = np.stack([np.full((n, 128), float(h)) for h in range(hkv)], axis=1)
    q = np.zeros((hkv * g_, 128))
    o = attention.decode_attention(q, kh, vh, np.stack([np.eye(128)] * hkv), g_)
    assert o[:, 0].tolist() == [0, 0, 1, 1, 2, 2]


def test_unquantized_identity_path_equals_reference():
    g = np.random.default_rng(4)
    k = g.standard_normal((40, 2, 128))
    v = g.standard_normal((40, 2, 128))
    q = g.standard_normal((4, 128))
    a = attention.decode_attention(q, k, v, np.stack([np.eye(128)] * 2), 2)
    b = attention.reference_attention(q, k, v, 2)
    assert np.abs(a - b).max() < 1e-13


def test_causal_attention_positions():
    g = np.random.default_rng(5)
    n, nq = 12, 3
    k = g.standard_normal((n, 1, 128))
    v = g.standard_normal((n, 1, 128))
    q = g.standard_normal((nq, 2, 128))
    o = attention.causal_attention(q, k, v, 2)
    for i in range(nq):
        t = n - nq + i
        ref = attention.reference_attention(q[i], k[: t + 1], v[: t + 1], 2)
        assert np.abs(o[i] - ref).max() < 1e-13
    # the last position sees every token
    assert np.abs(o[-1] - attention.reference_attention(q[-1], k, v, 2)).max() < 1e-13


def test_cache_read_path_feeds_attention():
    """Paged write + read + attention equals attention on directly quantized tensors."""
    g = np.random.default_rng(6)
    h, p, n = 2, 16, 45
    k = g.standard_normal((n, h, 128))
    v = g.standard_normal((n, h, 128))
    rk = np.stack([rotations.signed_hadamard(np.where(g.random(128) < .5, -1., 1.)) for _ in range(h)])
    mu = k.mean(axis=0)
    pool = np.zeros(cache.pool_bytes(4, h, p), np.uint8)
    table = np.array([3, 1, 0], np.int32)
    cache.write_tokens(pool, h, p, table, 0, cache.encode_tokens(k, v, rk, rk, mu, 1.0, 1.0))
    kh, vh = cache.dequantized_sequence(pool, h, p, table, n)
    q = g.standard_normal((4, 128))
    o = attention.decode_attention(q, kh, vh, rk, 2)
    kd = quant.quant_dequant(np.einsum("thc,hcd->thd", k - mu, rk), 1.0)
    vd = quant.quant_dequant(np.einsum("thc,hcd->thd", v, rk), 1.0)
    assert np.abs(o - attention.decode_attention(q, kd, vd, rk, 2)).max() < 1e-13
