"""GPU parity of the BF16 sink / recent windows: the window records written by
kvq_window_append byte for byte against the oracle, and kvq_decode_attention_win
against the oracle's windowed readout."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _mu(case):
    import oracle
    return oracle.cache.key_mean(case.calibration_keys()).astype(np.float32)


def _gpu_window(g, win_sizes):
    kvq, torch = g.kvq, g.torch
    s, r = win_sizes
    buf = torch.zeros(kvq.Window.buffer_bytes(g.case.n_seqs, g.case.n_kv_heads, s, r) or 16, dtype=torch.uint8,
                      device="cuda")
    return kvq.Window(s, r, buf)


def _append_windows(g, win, mu, chunks):
    """kvq_window_append of every sequence's tokens in the given chunk split (list of cut fractions)."""
    c = g.case
    kv = [c.kv(b) for b in range(c.n_seqs)]
    bounds = [np.unique(np.concatenate([[0], (np.asarray(chunks) * n).round().astype(int), [n]]))
              for n in g.lengths]
    n_steps = max(len(b) - 1 for b in bounds)
    mu_dev = gu.dev(mu)
    for ci in range(n_steps):
        ks, vs, cu, start = [], [], [0], []
        for b in range(c.n_seqs):
            bb = bounds[b]
            lo, hi = (bb[ci], bb[ci + 1]) if ci + 1 < len(bb) else (bb[-1], bb[-1])
            ks.append(kv[b][0][lo:hi])
            vs.append(kv[b][1][lo:hi])
            cu.append(cu[-1] + (hi - lo))
            start.append(lo)
        k = np.concatenate(ks)
        v = np.concatenate(vs)
        if len(k) == 0:
            continue
        g.kvq.kvq_window_append(g.layout, gu.dev(k, c.dtype), gu.dev(v, c.dtype), gu.dev_i32(cu), gu.dev_i32(start),
                                mu_dev, win)
    g.torch.cuda.synchronize()
    return bounds


def _oracle_windows(g, win_sizes, mu, bounds):
    import oracle
    s, r = win_sizes
    c = g.case
    regions = []
    for b in range(c.n_seqs):
        k, v = c.kv(b)
        reg = np.zeros((c.n_kv_heads, oracle.window.region_bytes(s, r)), np.uint8)
        bb = bounds[b]
        for lo, hi in zip(bb[:-1], bb[1:]):
            oracle.window.write_window(reg, k[lo:hi], v[lo:hi], int(lo), s, r, mu)
        regions.append(reg)
    return regions


WRITE_CASES = [
    # hkv, lengths, rot, dtype, (sink, recent), chunk cuts
    (2, [300, 77], "dense", "bf16", (64, 256), [0.5]),
    (1, [1000], "signed_hadamard", "f32", (64, 40), [0.1, 0.2, 0.95]),
    (4, [129, 64, 5], "identity", "f32", (128, 16), []),
    (2, [700, 333], "dense", "f32", (0, 64), [0.9, 0.901, 0.91, 0.999]),
    (3, [90, 200], "signed_hadamard", "bf16", (64, 0), [0.3]),
]


@pytest.mark.parametrize("hkv,lengths,rot,dtype,win_sizes,cuts", WRITE_CASES, ids=lambda v: str(v))
def test_window_records_match_the_oracle_bytes(hkv, lengths, rot, dtype, win_sizes, cuts):
    import oracle
    case = W.decode_case(41, lengths, 2 * hkv, hkv, 128, rot, dtype, n_cal=128)
    g = gu.GpuCase(case)
    mu = _mu(case)
    win = _gpu_window(g, win_sizes)
    bounds = _append_windows(g, win, mu, cuts)
    g.kvq.kvq_device_check()
    s, r = win_sizes
    per = oracle.window.region_bytes(s, r)
    got = win.buf.cpu().numpy()[: case.n_seqs * hkv * per].reshape(case.n_seqs, hkv, per)
    want = np.stack(_oracle_windows(g, win_sizes, mu, bounds))
    # one fp32 subtraction and bf16 roundings on both sides: bit-exact, no exemptions
    assert np.array_equal(got, want), f"{int((got != want).sum())} window bytes differ"


DECODE_CASES = [
    # hq, hkv, page, lengths, rot, dtype, (sink, recent), splits
    (4, 1, 16, [1, 63, 64, 65, 300, 321, 1000], "dense", "bf16", (64, 256), 0),
    (8, 2, 8, [257, 0, 3, 400], "signed_hadamard", "f32", (64, 40), 3),
    (16, 2, 16, [2049, 600], "dense", "bf16", (128, 24), 7),
    (2, 2, 16, [500, 37], "identity", "f32", (0, 16), 0),
    (32, 4, 16, [1000, 777], "signed_hadamard", "bf16", (64, 0), 0),
    (16, 16, 8, [100, 90], "dense", "f32", (64, 256), 1),
]


@pytest.mark.parametrize("hq,hkv,page,lengths,rot,dtype,win_sizes,splits", DECODE_CASES, ids=lambda v: str(v))
def test_windowed_decode_matches_the_oracle(hq, hkv, page, lengths, rot, dtype, win_sizes, splits):
    import oracle
    case = W.decode_case(42, lengths, hq, hkv, 128, rot, dtype, page_tokens=page, clip_k=0.96, clip_v=0.92, n_cal=256)
    g = gu.GpuCase(case)
    mu = _mu(case)
    ora_pool, _ = g.oracle_pool()
    pool = g.torch.from_numpy(ora_pool).cuda()
    bounds = [np.array([0, n]) for n in g.lengths]
    regions = _oracle_windows(g, win_sizes, mu, bounds)
    win = _gpu_window(g, win_sizes)
    flat = np.concatenate([reg.reshape(-1) for reg in regions])
    if flat.size:
        win.buf[: flat.size] = g.torch.from_numpy(flat).cuda()
    q = case.queries()
    max_len = int(g.lengths.max())
    kvq = g.kvq
    ws = g.torch.empty(kvq.kvq_decode_workspace_size_win(g.layout, case.n_seqs, max_len, win, splits),
                       dtype=g.torch.uint8, device="cuda")
    out = g.torch.full((case.n_seqs, hq, 128), float("nan"), device="cuda")
    kvq.kvq_decode_attention_win(g.layout, gu.dev(q, dtype), gu.dev_i32(g.lengths), max_len, g.table, g.rot_k,
                                 g.rot_v, pool, win, ws, out, n_splits=splits)
    kvq.kvq_device_check()
    got = out.cpu().numpy()
    s, r = win_sizes
    for b in range(case.n_seqs):
        n = int(g.lengths[b])
        if n == 0:
            assert np.all(got[b] == 0)
            continue
        kh, vh = oracle.cache.dequantized_sequence(ora_pool, hkv, page, case.block_table[b], n)
        wp, wk, wv = oracle.window.read_window(regions[b], n, s, r)
        ref = oracle.window.decode_attention_windowed(q[b], kh, vh, wp, wk, wv, g.r_k, g.r_v, case.gqa, n, s, r)
        err = gu.out_err(got[b], ref)
        assert np.isfinite(got[b]).all() and err <= gu.OUT_TOL, (b, n, err)


def test_end_to_end_windowed_steps():
    """Prefill chunk, then single-token steps that walk the recent ring around;
    both the INT2 pages and the window records written by the GPU."""
    import oracle
    lengths = [700, 410]
    case = W.decode_case(43, lengths, 8, 2, 128, "dense", "bf16", clip_k=0.96, clip_v=0.92, n_cal=256)
    g = gu.GpuCase(case)
    mu = _mu(case)
    sizes = (64, 40)
    win = _gpu_window(g, sizes)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    cuts = [0.8] + [0.8 + i / 1000 for i in range(1, 60)]  # many small appends near the end
    bounds = _append_windows(g, win, mu, cuts)
    regions = _oracle_windows(g, sizes, mu, bounds)
    got_buf = win.buf.cpu().numpy()
    per = oracle.window.region_bytes(*sizes)
    assert np.array_equal(got_buf.reshape(case.n_seqs, 2, per), np.stack(regions))
    q = case.queries()
    max_len = int(g.lengths.max())
    kvq = g.kvq
    ws = g.torch.empty(kvq.kvq_decode_workspace_size_win(g.layout, case.n_seqs, max_len, win), dtype=g.torch.uint8,
                       device="cuda")
    out = g.torch.empty((case.n_seqs, 8, 128), device="cuda")
    kvq.kvq_decode_attention_win(g.layout, gu.dev(q, "bf16"), gu.dev_i32(g.lengths), max_len, g.table, g.rot_k,
                                 g.rot_v, pool, win, ws, out)
    got = out.cpu().numpy()
    ora_pool, _ = g.oracle_pool()
    for b in range(case.n_seqs):
        n = lengths[b]
        kh, vh = oracle.cache.dequantized_sequence(ora_pool, 2, case.page_tokens, case.block_table[b], n)
        wp, wk, wv = oracle.window.read_window(regions[b], n, *sizes)
        ref = oracle.window.decode_attention_windowed(q[b], kh, vh, wp, wk, wv, g.r_k, g.r_v, case.gqa, n, *sizes)
        assert gu.out_err(got[b], ref) <= gu.OUT_TOL


def test_empty_window_is_the_plain_decode_and_splits_agree():
    case = W.decode_case(44, [3000, 1234], 8, 2, 128, "signed_hadamard", "bf16", n_cal=128)
    g = gu.GpuCase(case)
    ora_pool, _ = g.oracle_pool()
    pool = g.torch.from_numpy(ora_pool).cuda()
    q = case.queries()
    plain = g.gpu_decode(pool, q, n_splits=5)
    kvq = g.kvq
    win0 = kvq.Window(0, 0, None)
    ws = g.torch.empty(kvq.kvq_decode_workspace_size_win(g.layout, 2, 3000, win0, 5), dtype=g.torch.uint8,
                       device="cuda")
    out = g.torch.empty((2, 8, 128), device="cuda")
    kvq.kvq_decode_attention_win(g.layout, gu.dev(q, "bf16"), gu.dev_i32(g.lengths), 3000, g.table, g.rot_k,
                                 g.rot_v, pool, win0, ws, out, n_splits=5)
    assert np.array_equal(out.cpu().numpy(), plain)
    # with windows, the split count changes only the fp32 accumulation order
    import oracle
    mu = _mu(case)
    sizes = (64, 256)
    regions = _oracle_windows(g, sizes, mu, [np.array([0, n]) for n in g.lengths])
    win = _gpu_window(g, sizes)
    win.buf[:] = g.torch.from_numpy(np.concatenate([r.reshape(-1) for r in regions])).cuda()
    res = []
    for sp in (1, 5, 64):
        ws = g.torch.empty(kvq.kvq_decode_workspace_size_win(g.layout, 2, 3000, win, sp), dtype=g.torch.uint8,
                           device="cuda")
        kvq.kvq_decode_attention_win(g.layout, gu.dev(q, "bf16"), gu.dev_i32(g.lengths), 3000, g.table, g.rot_k,
                                     g.rot_v, pool, win, ws, out, n_splits=sp)
        res.append(out.cpu().numpy())
    assert gu.normwise_err(res[1], res[0]) < 5e-5 and gu.normwise_err(res[2], res[0]) < 5e-5


STEP_CASES = [
    # hq, hkv, page, lengths after the step, rot, dtype, (sink, recent), clips
    (8, 2, 16, [1, 40, 64, 65, 300, 0, 333], "dense", "bf16", (64, 40), (0.96, 0.92)),
    (32, 8, 8, [3000] * 6 + [2900], "dense", "bf16", (64, 256), (0.96, 0.92)),
    (16, 4, 16, [100, 257, 1000], "signed_hadamard", "f32", (64, 0), (1.0, 0.9)),
    (8, 2, 16, [10, 50, 70], "identity", "bf16", (0, 16), (0.9, 0.9)),
]


@pytest.mark.parametrize("hq,hkv,page,lengths,rot,dtype,win_sizes,clips", STEP_CASES, ids=lambda v: str(v))
def test_windowed_step_equals_separate_appends_and_the_oracle(hq, hkv, page, lengths, rot, dtype, win_sizes, clips):
    """kvq_decode_step_win against kvq_quantize_append + kvq_window_append +
    kvq_decode_attention_win on the same history: pools, window records and outputs
    equal bit for bit; the readout against the oracle's windowed decode."""
    import oracle
    case = W.decode_case(45, lengths, hq, hkv, 128, rot, dtype, page_tokens=page, clip_k=clips[0], clip_v=clips[1],
                         spare_blocks=2, n_cal=256)
    g = gu.GpuCase(case)
    kvq, torch = g.kvq, g.torch
    mu = _mu(case)
    full = g.lengths.copy()
    hist = np.maximum(full - 1, 0)
    # history: every token but the last, in the pool and the windows
    g.lengths = hist
    pool_a = g.new_pool()
    if hist.sum():
        g.gpu_append_all(pool_a)
    win_a = _gpu_window(g, win_sizes)
    if hist.sum():
        _append_windows(g, win_a, mu, [])
    g.lengths = full
    pool_b = pool_a.clone()
    win_b = kvq.Window(win_sizes[0], win_sizes[1], win_a.buf.clone())
    kv = [case.kv(b) for b in range(case.n_seqs)]
    zero = np.zeros((hkv, 128), np.float32)
    k_new = np.stack([kv[b][0][full[b] - 1] if full[b] else zero for b in range(case.n_seqs)])
    v_new = np.stack([kv[b][1][full[b] - 1] if full[b] else zero for b in range(case.n_seqs)])
    has = full > 0
    cu = gu.dev_i32(np.concatenate([[0], np.cumsum(has)]))
    start = gu.dev_i32(hist)
    kn, vn = gu.dev(k_new, dtype), gu.dev(v_new, dtype)
    q = gu.dev(case.queries(), dtype)
    lens = gu.dev_i32(full)
    max_len = int(full.max())
    mu_dev = gu.dev(mu)
    ws = torch.empty(kvq.kvq_decode_workspace_size_win(g.layout, case.n_seqs, max_len, win_a), dtype=torch.uint8,
                     device="cuda")
    # separate calls
    kvq.kvq_quantize_append(g.layout, gu.dev(k_new[has], dtype), gu.dev(v_new[has], dtype), cu, start, g.table,
                            g.rot_k, g.rot_v, g.mu_rot_dev, case.clip_k, case.clip_v, pool_a)
    kvq.kvq_window_append(g.layout, gu.dev(k_new[has], dtype), gu.dev(v_new[has], dtype), cu, start, mu_dev, win_a)
    out_a = torch.full((case.n_seqs, hq, 128), float("nan"), device="cuda")
    kvq.kvq_decode_attention_win(g.layout, q, lens, max_len, g.table, g.rot_k, g.rot_v, pool_a, win_a, ws, out_a)
    # the fused step
    out_b = torch.full_like(out_a, float("nan"))
    kvq.kvq_decode_step_win(g.layout, q, kn, vn, lens, max_len, g.table, g.rot_k, g.rot_v, g.mu_rot_dev, mu_dev,
                            case.clip_k, case.clip_v, pool_b, win_b, ws, out_b)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(win_a.buf, win_b.buf)
    assert torch.equal(out_a, out_b)
    # the oracle: windows of every token, windowed readout over the pool
    ora_pool, _ = g.oracle_pool()
    regions = _oracle_windows(g, win_sizes, mu, [np.array([0, n]) for n in full])
    got = out_b.cpu().numpy()
    s, r = win_sizes
    for b in range(case.n_seqs):
        n = int(full[b])
        if n == 0:
            assert np.all(got[b] == 0)
            continue
        kh, vh = oracle.cache.dequantized_sequence(ora_pool, hkv, page, case.block_table[b], n)
        wp, wk, wv = oracle.window.read_window(regions[b], n, s, r)
        ref = oracle.window.decode_attention_windowed(case.queries()[b], kh, vh, wp, wk, wv, g.r_k, g.r_v, case.gqa,
                                                      n, s, r)
        assert gu.out_err(got[b], ref) <= gu.OUT_TOL, (b, n, gu.out_err(got[b], ref))
