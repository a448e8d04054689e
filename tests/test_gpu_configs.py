"""The five named workloads on the GPU, checked against the fp64 oracle.

Small workloads are compared in full; full-size ones (16 x 32K, 128K context,
64 ragged sequences) are built and decoded in full on the GPU, and the oracle
recomputes a seeded sample of sequences one by one."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def build_full_cache(g, pool):
    """Append every sequence with one kvq_quantize_append call per sequence."""
    c = g.case
    for b in range(c.n_seqs):
        k, v = c.kv(b)
        n = int(g.lengths[b])
        g.kvq.kvq_quantize_append(g.layout, gu.dev(k[:n], c.dtype), gu.dev(v[:n], c.dtype), gu.dev_i32([0, n]),
                                  gu.dev_i32([0]), g.table[b:b + 1].contiguous(), g.rot_k, g.rot_v, g.mu_rot_dev,
                                  c.clip_k, c.clip_v, pool)
    g.torch.cuda.synchronize()
    g.kvq.kvq_device_check()


def oracle_seq(g, b, n=None):
    import oracle
    c = g.case
    k, v = c.kv(b)
    n = int(g.lengths[b]) if n is None else n
    enc = oracle.cache.encode_tokens(k[:n], v[:n], g.r_k, g.r_v, None, c.clip_k, c.clip_v, mu_rot=g.mu_rot)
    pool = np.zeros(oracle.cache.pool_bytes(c.num_blocks, c.n_kv_heads, c.page_tokens), np.uint8)
    oracle.cache.write_tokens(pool, c.n_kv_heads, c.page_tokens, c.block_table[b], 0, enc)
    return pool, enc


def check_sampled(g, gpool_np, q, got, seqs):
    import oracle
    c = g.case
    for b in seqs:
        pool_b, enc = oracle_seq(g, b)
        lens = [0] * c.n_seqs
        lens[b] = int(g.lengths[b])
        encs = [None] * c.n_seqs
        encs[b] = enc
        gu.compare_codes(gpool_np, pool_b, c.n_kv_heads, c.page_tokens, c.block_table, lens, encs,
                         (c.clip_k, c.clip_v), label=f"{c.name} seq {b}")
        kh, vh = oracle.cache.dequantized_sequence(pool_b, c.n_kv_heads, c.page_tokens, c.block_table[b], lens[b])
        ref = oracle.attention.decode_attention(q[b], kh, vh, g.r_k, c.gqa)
        assert gu.out_err(got[b], ref) <= gu.OUT_TOL, (b, gu.out_err(got[b], ref))


def test_tiny_single_head_end_to_end():
    """1 query, 512 fp32 tokens, signed-Hadamard R, clip 1.0: y and NMSE vs the oracle."""
    import oracle
    c = W.tiny_single_head()
    g = gu.GpuCase(c)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    q = c.queries()
    o = g.gpu_decode(pool, q)
    torch = g.torch
    w = c.w_o()
    wf = torch.empty(128, 128, device="cuda")
    g.kvq.kvq_fold_wo(gu.dev(w), 1, 1, g.rot_v, wf)
    y = torch.empty(1, 128, device="cuda")
    g.kvq.kvq_out_proj(gu.dev(o).reshape(1, -1), wf, y)
    y = y.cpu().numpy()
    ora_pool, _ = g.oracle_pool()
    o_ref_q = g.oracle_decode(ora_pool, q)[0]
    y_o = oracle.output.out_proj(o_ref_q[None], oracle.output.fold_wo(w, g.r_v, 1))
    k, v = c.kv(0)
    y_ref = oracle.output.out_proj(oracle.attention.reference_attention(q[0], k, v, 1)[None], w)
    assert gu.out_err(y, y_o) <= gu.OUT_TOL
    n_gpu, n_ora = oracle.output.nmse(y, y_ref), oracle.output.nmse(y_o, y_ref)
    assert abs(n_gpu - n_ora) <= gu.NMSE_TOL * n_ora
    print(f"tiny: NMSE gpu {n_gpu:.6g} oracle {n_ora:.6g}")


def test_envelope_selection_then_fresh_queries():
    """Evaluation page envelope: select (R, c) on one calibration query, then score
    10 fresh queries through the paged GPU path (quantize-append, decode, W_O)."""
    import oracle
    from test_gpu_calib import run_gpu_calib
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    cc = W.envelope_calibration()
    mu = oracle.cache.key_mean(cc.k).astype(np.float32)
    nm, _ = run_gpu_calib(cc, mu)
    ci, ki = oracle.calib.select(nm)[0]
    spec = cc.cands[ci]
    clip = cc.clips[ki]
    hkv, page = 4, 16
    table = np.arange(4096 // page, dtype=np.int32)[None]
    lay = kvq.make_layout(page, hkv, hkv, 4096 // page, 4096 // page)
    r = oracle.rotations.rot_matrices(spec, hkv)
    mu_rot = np.einsum("hc,hcd->hd", mu.astype(np.float64), r).astype(np.float32)
    drot = kvq.DeviceRot.from_spec(spec)
    pool = torch.zeros(kvq.kvq_pool_bytes(lay), dtype=torch.uint8, device="cuda")
    kvq.kvq_quantize_append(lay, gu.dev(cc.k), gu.dev(cc.v), gu.dev_i32([0, 4096]), gu.dev_i32([0]), gu.dev_i32(table),
                            drot, drot, gu.dev(mu_rot), clip, clip, pool)
    wf = torch.empty(128, 512, device="cuda")
    kvq.kvq_fold_wo(gu.dev(cc.w_o), 4, 4, drot, wf)
    nq = cc.fresh_q.shape[0]
    ws = torch.empty(kvq.kvq_decode_workspace_size(lay, nq, 4096), dtype=torch.uint8, device="cuda")
    # the 10 fresh queries as 10 sequences sharing one block table row
    lay10 = kvq.make_layout(page, hkv, hkv, 4096 // page, 4096 // page)
    table10 = gu.dev_i32(np.repeat(table, nq, axis=0))
    o = torch.empty(nq, 4, 128, device="cuda")
    kvq.kvq_decode_attention(lay10, gu.dev(cc.fresh_q), gu.dev_i32([4096] * nq), 4096, table10, drot, pool, ws, o)
    y = torch.empty(nq, 128, device="cuda")
    kvq.kvq_out_proj(o.reshape(nq, -1), wf, y)
    y = y.cpu().numpy()
    # oracle: same selected (R, c), fp64 pipeline, unquantized reference
    enc = oracle.cache.encode_tokens(cc.k, cc.v, r, r, None, clip, clip, mu_rot=mu_rot)
    kh = oracle.quant.dequantize_groups(enc["ck"], enc["sk"], enc["zk"])
    vh = oracle.quant.dequantize_groups(enc["cv"], enc["sv"], enc["zv"])
    wfo = oracle.output.fold_wo(cc.w_o, r, 1)
    n_gpu, n_ora = [], []
    for i in range(nq):
        y_o = oracle.output.out_proj(oracle.attention.decode_attention(cc.fresh_q[i], kh, vh, r, 1)[None], wfo)
        y_ref = oracle.output.out_proj(oracle.attention.reference_attention(cc.fresh_q[i], cc.k, cc.v, 1)[None], cc.w_o)
        assert gu.out_err(y[i], y_o[0]) <= gu.OUT_TOL
        n_gpu.append(oracle.output.nmse(y[i], y_ref[0]))
        n_ora.append(oracle.output.nmse(y_o[0], y_ref[0]))
    n_gpu, n_ora = np.array(n_gpu), np.array(n_ora)
    gu.assert_nmse_close(n_gpu, n_ora, "fresh-query nmse")
    m, sd = oracle.output.mean_popsd(n_gpu)
    tm, tsd = oracle.output.threshold_rate(n_gpu)
    print(f"envelope: selected candidate {ci} clip {clip}: NMSE {m:.6f} +- {sd:.6f}, threshold {tm:.2f} +- {tsd:.2f}")


def test_gqa8b_32k_full_size_sampled():
    """16 x 32,768 tokens, 32/8 heads, dense R: full GPU cache + decode; the oracle
    re-derives sequences 0 and 15."""
    c = W.gqa8b_32k()
    g = gu.GpuCase(c)
    pool = g.new_pool()
    build_full_cache(g, pool)
    q = c.queries()
    got = g.gpu_decode(pool, q)
    assert np.isfinite(got).all()
    check_sampled(g, pool.cpu().numpy(), q, got, [0, 15])


def test_long4b_128k_with_prefill_chunk():
    """131,072 tokens, signed Hadamard, clip 0.9; the last 4,096 tokens arrive as a
    prefill-chunk append at a page-aligned offset."""
    c = W.long4b_128k(n_seqs=1)
    g = gu.GpuCase(c)
    pool = g.new_pool()
    k, v = c.kv(0)
    n = c.seq_lens[0]
    hist = n - 4096
    for lo, hi in ((0, hist), (hist, n)):
        g.kvq.kvq_quantize_append(g.layout, gu.dev(k[lo:hi], "bf16"), gu.dev(v[lo:hi], "bf16"), gu.dev_i32([0, hi - lo]),
                                  gu.dev_i32([lo]), g.table, g.rot_k, g.rot_v, g.mu_rot_dev, c.clip_k, c.clip_v, pool)
    g.torch.cuda.synchronize()
    g.kvq.kvq_device_check()
    q = c.queries()
    got = g.gpu_decode(pool, q)
    check_sampled(g, pool.cpu().numpy(), q, got, [0])


def test_serve14b_ragged_step():
    """64 ragged contexts, 40/10 heads, dense R: build, then one decode step that
    appends one token per sequence and decodes at the new length."""
    c = W.serve14b_ragged()
    new_lens = c.seq_lens + 1
    c2 = W.decode_case(c.seed, new_lens, 40, 10, 5120, "dense", "bf16", n_cal=2560, name=c.name)
    g = gu.GpuCase(c2)
    pool = g.new_pool()
    # history: the first L_b tokens of each sequence (drawn from the same per-sequence stream)
    g.lengths = c.seq_lens.copy()
    build_full_cache(g, pool)
    # step: one new token per sequence at position L_b
    ks, vs = [], []
    for b in range(c2.n_seqs):
        k, v = c2.kv(b)
        ks.append(k[c.seq_lens[b]:c.seq_lens[b] + 1])
        vs.append(v[c.seq_lens[b]:c.seq_lens[b] + 1])
    g.kvq.kvq_quantize_append(g.layout, gu.dev(np.concatenate(ks), "bf16"), gu.dev(np.concatenate(vs), "bf16"),
                              gu.dev_i32(np.arange(c2.n_seqs + 1)), gu.dev_i32(c.seq_lens), g.table, g.rot_k, g.rot_v,
                              g.mu_rot_dev, c2.clip_k, c2.clip_v, pool)
    g.lengths = new_lens
    q = c2.queries()
    got = g.gpu_decode(pool, q)
    g.kvq.kvq_device_check()
    check_sampled(g, pool.cpu().numpy(), q, got, [0, 31, 63])


def test_serve14b_calibration_sampled():
    """16 dense candidates x 5 clips x 10 heads over 2,560 calibration tokens and 64
    causal query positions; the oracle recomputes three candidates."""
    import oracle
    from test_gpu_calib import run_gpu_calib
    cc = W.serve14b_calibration()
    mu = oracle.cache.key_mean(cc.k).astype(np.float32)
    nm, ref = run_gpu_calib(cc, mu)
    sample = [0, 7, 15]
    sub = W.CalibCase(cc.seed, cc.n_tok, cc.n_qpos, cc.n_kv_heads, cc.gqa, cc.d_model, cc.dtype, cc.k, cc.v, cc.q,
                      cc.w_o, [cc.cands[i] for i in sample], cc.clips, cc.joint)
    mats = [oracle.rotations.rot_matrices(x, cc.n_kv_heads) for x in sub.cands]
    nm_o, _, ref_o = oracle.calib.calib_sweep(sub.q, sub.k, sub.v, sub.w_o, mats, sub.clips, mu, sub.gqa, False)
    gu.assert_nmse_close(ref, ref_o, "ref")
    gu.assert_nmse_close(nm[sample], nm_o, "serve14b nmse")


def test_gqa8b_32k_table_a_windows_sampled():
    """Table A in full at the 8B-class decode shape: 16 x 32,768 tokens, 8-token pages,
    clips 0.96 / 0.92, 64 sink + 256 recent BF16 tokens; the whole cache and the window
    records written by the GPU, the windowed decode over all of it; the oracle re-derives
    sequences 0 and 15 (INT2 pages, window records, windowed readout)."""
    import oracle
    c = W.gqa8b_32k(page_tokens=8, clip_k=0.96, clip_v=0.92)
    g = gu.GpuCase(c)
    kvq, torch = g.kvq, g.torch
    pool = g.new_pool()
    build_full_cache(g, pool)
    s_w, r_w = 64, 256
    mu = oracle.cache.key_mean(c.calibration_keys()).astype(np.float32)
    mu_dev = gu.dev(mu)
    per = kvq.Window.buffer_bytes(1, c.n_kv_heads, s_w, r_w)
    buf = torch.zeros(per * c.n_seqs, dtype=torch.uint8, device="cuda")
    L = int(c.seq_lens[0])
    spans = ((0, s_w), (L - r_w, L))
    for b in range(c.n_seqs):
        k, v = c.kv(b)
        row = kvq.Window(s_w, r_w, buf[b * per:(b + 1) * per])
        for lo, hi in spans:  # the sink, then the recent tokens (window tokens at length L)
            kvq.kvq_window_append(g.layout, gu.dev(k[lo:hi], "bf16"), gu.dev(v[lo:hi], "bf16"),
                                  gu.dev_i32([0, hi - lo]), gu.dev_i32([lo]), mu_dev, row)
    torch.cuda.synchronize()
    win = kvq.Window(s_w, r_w, buf)
    ws = torch.empty(kvq.kvq_decode_workspace_size_win(g.layout, c.n_seqs, L, win), dtype=torch.uint8, device="cuda")
    out = torch.full((c.n_seqs, c.n_q_heads, 128), float("nan"), device="cuda")
    q = c.queries()
    kvq.kvq_decode_attention_win(g.layout, gu.dev(q, "bf16"), gu.dev_i32(g.lengths), L, g.table, g.rot_k, g.rot_v,
                                 pool, win, ws, out)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    gpool = pool.cpu().numpy()
    gbuf = buf.cpu().numpy()
    for b in (0, 15):
        pool_b, enc = oracle_seq(g, b)
        lens = [0] * c.n_seqs
        lens[b] = L
        encs = [None] * c.n_seqs
        encs[b] = enc
        gu.compare_codes(gpool, pool_b, c.n_kv_heads, c.page_tokens, c.block_table, lens, encs, (c.clip_k, c.clip_v),
                         label=f"table A seq {b}")
        k, v = c.kv(b)
        reg = np.zeros((c.n_kv_heads, oracle.window.region_bytes(s_w, r_w)), np.uint8)
        for lo, hi in spans:
            oracle.window.write_window(reg, k[lo:hi], v[lo:hi], lo, s_w, r_w, mu)
        assert np.array_equal(gbuf[b * per:(b + 1) * per].reshape(reg.shape), reg), f"window records of seq {b}"
        kh, vh = oracle.cache.dequantized_sequence(pool_b, c.n_kv_heads, c.page_tokens, c.block_table[b], L)
        wp, wk, wv = oracle.window.read_window(reg, L, s_w, r_w)
        ref = oracle.window.decode_attention_windowed(q[b], kh, vh, wp, wk, wv, g.r_k, g.r_v, c.gqa, L, s_w, r_w)
        assert gu.out_err(got[b], ref) <= gu.OUT_TOL, (b, gu.out_err(got[b], ref))
