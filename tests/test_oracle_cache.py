"""Pins for oracle.cache: page layout, write/read, payload and storage constants."""
import json
import os

import numpy as np

from oracle import cache, quant, rotations
from conftest import GOLDEN


def test_record_layout_hand_offsets():
    p, h = 16, 2
    assert cache.record_bytes(p) == 1152 and cache.record_bytes(8) == 576
    pool = np.zeros(cache.pool_bytes(3, h, p), np.uint8)
    x = np.zeros((1, h, 128))
    x[0, 1, 0] = 3.0  # head 1, K: channel 0 -> code 3 (range [0, 3])
    v = np.zeros((1, h, 128))
    v[0, 0, 127] = -3.0  # head 0, V: channel 127 is the min -> code 0, others code 3
    enc = cache.encode_tokens(x, v, np.stack([np.eye(128)] * h), np.stack([np.eye(128)] * h), None, 1.0, 1.0)
    table = np.array([2, 0], np.int32)
    cache.write_tokens(pool, h, p, table, 17, enc)  # pos 17 -> page 1 -> block 0, slot 1
    rec = pool.reshape(3, h, 1152)
    # head 1 K codes of slot 1: byte 0 holds channel 0 = code 3 in bits 0..1
    assert rec[0, 1, 32 * 1 + 0] == 3 and rec[0, 1, 32:64].sum() == 3
    # head 1 K meta at 1024 + 4*1: scale fp16(1.0) = 0x3C00, zero 0
    assert rec[0, 1, 1028:1032].tolist() == [0x00, 0x3C, 0x00, 0x00]
    # head 0 V codes at 512 + 32: channels 0..126 code 3, channel 127 code 0
    vb = rec[0, 0, 512 + 32: 512 + 64]
    assert vb[:31].tolist() == [255] * 31 and vb[31] == 0b00111111
    # head 0 V meta at 1088 + 4: scale 1.0, zero -3.0 = 0xC200
    assert rec[0, 0, 1092:1096].tolist() == [0x00, 0x3C, 0x00, 0xC2]
    # nothing else written
    assert rec[1:].sum() == 0 and rec[2].sum() == 0
    touched = np.zeros_like(rec[0], bool)
    for hh, lo, hi in ((1, 32, 64), (1, 1028, 1032), (0, 512 + 32, 512 + 64), (0, 1092, 1096),
                       (0, 32, 64), (0, 1028, 1032), (1, 512 + 32, 512 + 64), (1, 1092, 1096)):
        touched[hh, lo:hi] = True
    assert rec[0][~touched].sum() == 0


def test_write_read_round_trip_across_pages():
    g = np.random.default_rng(0)
    h, p, n = 3, 8, 37
    k = g.standard_normal((n, h, 128))
    v = g.standard_normal((n, h, 128))
    rk = np.stack([rotations.expm_skew(g.normal(0, 0.05, (128, 128))) for _ in range(h)])
    rv = np.stack([rotations.signed_hadamard(np.where(g.random(128) < .5, -1., 1.)) for _ in range(h)])
    mu = g.standard_normal((h, 128))
    table = g.permutation(8).astype(np.int32)
    pool = np.zeros(cache.pool_bytes(8, h, p), np.uint8)
    enc = cache.encode_tokens(k, v, rk, rv, mu, 0.9, 0.95)
    cache.write_tokens(pool, h, p, table, 0, {kk: vv[:20] for kk, vv in enc.items()})
    cache.write_tokens(pool, h, p, table, 20, {kk: vv[20:] for kk, vv in enc.items()})
    r = cache.read_sequence(pool, h, p, table, n)
    for key in ("ck", "sk", "zk", "cv", "sv", "zv"):
        assert np.array_equal(r[key], enc[key]), key
    # the stored key is Q_2((k - mu) R_K) (Eq. 21)
    kh, _ = cache.dequantized_sequence(pool, h, p, table, n)
    xk = np.einsum("thc,hcd->thd", k - mu[None], rk)
    assert np.array_equal(kh, quant.quant_dequant(xk, 0.9))


def test_identity_rotation_cache_equals_plain_int2_bytes():
    g = np.random.default_rng(1)
    k = g.standard_normal((16, 1, 128)) * 3
    v = g.standard_normal((16, 1, 128))
    e = cache.encode_tokens(k, v, np.eye(128)[None], np.eye(128)[None], None, 1.0, 1.0)
    ck, sk, zk = quant.quantize_groups(k, 1.0)
    assert np.array_equal(quant.pack_codes(e["ck"]), quant.pack_codes(ck))
    assert np.array_equal(e["sk"], sk) and np.array_equal(e["zk"], zk)


def test_payload_bytes_of_the_evaluation_envelope():
    with open(os.path.join(GOLDEN, "evaluation_page.json")) as f:
        page = json.load(f)
    t, h, d = page["tokens"], page["kv_heads"], page["head_dim"]
    p = 16
    n_pages = t // p
    pool_total = cache.pool_bytes(n_pages, h, p)
    code_bytes = n_pages * h * 2 * 32 * p  # K and V code regions of every record
    assert code_bytes == t * h * d * 2 * 2 // 8 == page["packed_kv_bytes"]
    assert pool_total - code_bytes == t * h * 2 * 4 == 131072


def test_bits_per_element_and_storage_ratio():
    with open(os.path.join(GOLDEN, "paper_constants.json")) as f:
        c = json.load(f)
    g = c["group_size"]
    bits_int2 = 2 + 32 / g  # 2-bit code + (fp16 scale + fp16 zero) per group
    n = c["bpe_context"]
    w = c["sink_tokens"] + c["recent_tokens"]
    bpe = ((n - w) * bits_int2 + w * 16) / n
    assert round(bpe, 2) == c["bpe_reported"]
    assert 2 / 16 == c["int2_fraction_of_bf16"] and 2 / 4 == c["int2_fraction_of_int4"]


def test_key_mean_and_rotate_heads():
    k = np.arange(2 * 3 * 128, dtype=np.float64).reshape(2, 3, 128)
    mu = cache.key_mean(k)
    assert np.array_equal(mu, (k[0] + k[1]) / 2)
    r = np.stack([np.eye(128), 2 * np.eye(128)])
    x = np.ones((4, 128))
    y = cache.rotate_heads(x, r, heads_per_rot=2)  # heads 0,1 -> R0; 2,3 -> R1
    assert np.array_equal(y[:2], np.ones((2, 128))) and np.array_equal(y[2:], 2 * np.ones((2, 128)))


def test_rotate_then_subtract_form_equals_centre_then_rotate():
    # Eq. 20: (k - mu) R = k R - mu R
    g = np.random.default_rng(7)
    h = 2
    k = g.standard_normal((9, h, 128)) * 4
    v = g.standard_normal((9, h, 128))
    r = np.stack([rotations.expm_skew(g.normal(0, 0.05, (128, 128))) for _ in range(h)])
    mu = g.standard_normal((h, 128))
    a = cache.encode_tokens(k, v, r, r, mu, 1.0, 1.0)
    b = cache.encode_tokens(k, v, r, r, None, 1.0, 1.0, mu_rot=np.einsum("hc,hcd->hd", mu, r))
    assert np.abs(a["xk"] - b["xk"]).max() < 1e-12
