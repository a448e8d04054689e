"""Pins for oracle.window: bf16 rounding, window membership and layout, ring
contents after chunked appends, and the windowed readout on inputs that the
INT2 and BF16 paths both store losslessly (so it must equal plain attention)."""
import numpy as np
import pytest
import torch

from oracle import attention, cache, rotations, window

D = 128


def test_bf16_rounding_matches_torch_conversion():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(2000) * 1e-38).astype(np.float32),   # bf16 subnormal range
        (g.standard_normal(2000) * 1e37).astype(np.float32),
        # exact midpoints between neighbouring bf16 values: ties go to the even neighbour
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 + 2 ** -134, 3.0 + 2 ** -7],
                 np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = window.bf16_rne(x.astype(np.float64))
    assert np.array_equal(got, want)
    assert np.array_equal(window.bf16_bits(got),
                          torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    assert window.bf16_rne([1 + 2 ** -8])[0] == 1.0 and window.bf16_rne([1 + 3 * 2 ** -8])[0] == 1 + 2 ** -6


def test_membership_matches_brute_force():
    for sink in (0, 64, 128):
        for recent in (0, 8, 24, 256):
            for length in (0, 1, 7, 63, 64, 65, 100, 320, 321, 1000):
                want = sorted(p for p in range(length) if p < sink or p >= length - recent)
                assert window.window_positions(length, sink, recent).tolist() == want
                rest = sorted(set(range(length)) - set(want))
                assert window.int2_positions(length, sink, recent).tolist() == rest


def test_record_layout_is_a_bijection():
    sink, recent = 64, 24
    nbytes = window.region_bytes(sink, recent)
    assert nbytes == (64 + 24) * 512
    offs = [window.element_offset(s, part, np.arange(D)) for s in range(sink + recent) for part in (0, 1)]
    offs = np.concatenate(offs)
    assert np.array_equal(np.sort(offs), np.arange(0, nbytes, 2))
    # slot 9 = record 1, row 1: channel 0 (chunk 0) sits at chunk position 1 of the row
    assert window.element_offset(9, 0, 0) == 4096 + 256 + 16
    assert window.element_offset(9, 1, 8) == 4096 + 2048 + 256 + 0
    # ring slots: position p >= sink goes to sink + p mod recent
    assert window.slot_of([0, 63, 64, 87, 88, 1000], sink, recent).tolist() == [0, 63, 64 + 16, 64 + 15, 64 + 16, 64 + 16]


def test_ring_contents_after_chunked_appends():
    g = np.random.default_rng(1)
    h, sink, recent = 2, 64, 40
    total = 400
    k = g.standard_normal((total, h, D)).astype(np.float32).astype(np.float64) * 3
    v = g.standard_normal((total, h, D)).astype(np.float32).astype(np.float64)
    mu = g.standard_normal((h, D)).astype(np.float32).astype(np.float64)
    region = np.zeros((h, window.region_bytes(sink, recent)), np.uint8)
    pos = 0
    for n in (1, 70, 1, 1, 90, 3, 200, 1, 33):
        window.write_window(region, k[pos:pos + n], v[pos:pos + n], pos, sink, recent, mu)
        pos += n
        wp, wk, wv = window.read_window(region, pos, sink, recent)
        assert np.array_equal(wp, window.window_positions(pos, sink, recent))
        # the key: one fp32 subtraction rounded to bf16; the value: v rounded to bf16
        kk = torch.from_numpy((k[wp].astype(np.float32) - mu.astype(np.float32)[None])).to(torch.bfloat16)
        assert np.array_equal(wk, kk.to(torch.float64).numpy())
        vv = torch.from_numpy(v[wp].astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(wv, vv)


def _grid_group(g, n):
    """n rows of 128 values on a 4-level grid lo + i s (both levels 0 and 3 present),
    lo, s multiples of 1/8: INT2 with clip 1 stores them exactly."""
    lo = g.integers(-24, 0, (n, 1)) / 8.0
    s = g.integers(1, 12, (n, 1)) / 8.0
    i = g.integers(0, 4, (n, D))
    i[:, 0], i[:, 1] = 0, 3
    return lo + s * i


@pytest.mark.parametrize("sink,recent,length", [(0, 0, 150), (64, 40, 150), (64, 256, 150), (0, 16, 37),
                                                (128, 8, 500)])
def test_windowed_readout_equals_plain_attention_on_lossless_inputs(sink, recent, length):
    """Window tokens: k - mu and v exact in bf16; INT2 tokens: (k - mu) R_K and
    v R_V on the INT2 grid.  Both stores are then lossless, and the windowed
    readout, rotated back, must equal attention on the raw k, v (Eqs. 1-2, 24, 27)."""
    g = np.random.default_rng(sink + recent + length)
    hkv, gqa = 2, 2
    r_k = np.stack([rotations.expm_skew(g.normal(0, 0.05, (D, D))) for _ in range(hkv)])
    r_v = np.stack([rotations.expm_skew(g.normal(0, 0.05, (D, D))) for _ in range(hkv)])
    mu = g.integers(-16, 16, (hkv, D)) / 8.0
    win = np.zeros(length, bool)
    win[window.window_positions(length, sink, recent)] = True
    xk = np.where(win[:, None, None], g.integers(-40, 40, (length, hkv, D)) / 8.0,
                  _grid_group(g, length * hkv).reshape(length, hkv, D))
    xv = np.where(win[:, None, None], g.integers(-40, 40, (length, hkv, D)) / 8.0,
                  _grid_group(g, length * hkv).reshape(length, hkv, D))
    # window keys: k - mu = xk (unrotated); INT2 keys: (k - mu) R_K = xk
    k = np.where(win[:, None, None], xk, np.einsum("thd,hcd->thc", xk, r_k)) + mu[None]
    # window values: v = xv (stored as is); INT2 values: v R_V = xv
    v = np.where(win[:, None, None], xv, np.einsum("thd,hcd->thc", xv, r_v))
    q = g.standard_normal((hkv * gqa, D))

    enc = cache.encode_tokens(k, v, r_k, r_v, mu, 1.0, 1.0)
    k_hat = enc["zk"][..., None] + enc["sk"][..., None] * enc["ck"]
    v_hat = enc["zv"][..., None] + enc["sv"][..., None] * enc["cv"]
    ip = window.int2_positions(length, sink, recent)
    if len(ip):
        assert np.abs(k_hat[ip] - xk[ip]).max() < 1e-12 and np.abs(v_hat[ip] - xv[ip]).max() < 1e-12

    region = np.zeros((hkv, max(window.region_bytes(sink, recent), 1)), np.uint8)
    if sink + recent:
        window.write_window(region, k, v, 0, sink, recent, mu)
    wp, wk, wv = window.read_window(region, length, sink, recent)
    got = window.decode_attention_windowed(q, k_hat, v_hat, wp, wk, wv, r_k, r_v, gqa, length, sink, recent)
    ref = attention.reference_attention(q, k, v, gqa)
    back = np.einsum("jd,jcd->jc", got, r_v[np.arange(hkv * gqa) // gqa])  # o' R_V^T
    assert np.abs(back - ref).max() < 1e-11 * max(1.0, np.abs(ref).max())


def test_empty_windows_equal_plain_decode():
    g = np.random.default_rng(3)
    length, hkv, gqa = 90, 2, 4
    r_k = np.stack([rotations.expm_skew(g.normal(0, 0.05, (D, D))) for _ in range(hkv)])
    k_hat = g.standard_normal((length, hkv, D))
    v_hat = g.standard_normal((length, hkv, D))
    q = g.standard_normal((hkv * gqa, D))
    wp = np.zeros(0, np.int64)
    got = window.decode_attention_windowed(q, k_hat, v_hat, wp, np.zeros((0, hkv, D)), np.zeros((0, hkv, D)),
                                           r_k, r_k, gqa, length, 0, 0)
    assert np.array_equal(got, attention.decode_attention(q, k_hat, v_hat, r_k, gqa)) or \
        np.abs(got - attention.decode_attention(q, k_hat, v_hat, r_k, gqa)).max() < 1e-14


def test_windowed_readout_matches_brute_force_loops():
    """Pure-Python loops over a tiny mixed sequence: INT2 positions meet q' = q R_K,
    window positions meet the unrotated q; one softmax over all of them; window
    values enter the rotated-V readout as v R_V."""
    import math
    g = np.random.default_rng(4)
    length, sink, recent, hkv, gqa = 11, 0, 8, 1, 2
    r_k = rotations.expm_skew(g.normal(0, 0.3, (D, D)))[None]
    r_v = rotations.expm_skew(g.normal(0, 0.3, (D, D)))[None]
    q = g.standard_normal((gqa, D))
    k_hat = g.standard_normal((length, hkv, D))
    v_hat = g.standard_normal((length, hkv, D))
    wp = window.window_positions(length, sink, recent)
    wk = g.standard_normal((len(wp), hkv, D))
    wv = g.standard_normal((len(wp), hkv, D))
    got = window.decode_attention_windowed(q, k_hat, v_hat, wp, wk, wv, r_k, r_v, gqa, length, sink, recent)
    for j in range(gqa):
        qj = q[j].tolist()
        qr = [sum(qj[c] * r_k[0][c][d] for c in range(D)) for d in range(D)]
        logits, vals = [], []
        for p in range(length):
            if p in wp.tolist():
                i = wp.tolist().index(p)
                logits.append(sum(qj[d] * wk[i][0][d] for d in range(D)) / math.sqrt(D))
                vals.append([sum(wv[i][0][c] * r_v[0][c][d] for c in range(D)) for d in range(D)])
            else:
                logits.append(sum(qr[d] * k_hat[p][0][d] for d in range(D)) / math.sqrt(D))
                vals.append(v_hat[p][0])
        m = max(logits)
        e = [math.exp(a - m) for a in logits]
        z = sum(e)
        want = [sum(e[t] / z * vals[t][d] for t in range(length)) for d in range(D)]
        assert np.abs(got[j] - np.array(want)).max() < 1e-12
