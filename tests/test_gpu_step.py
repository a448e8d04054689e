"""GPU parity of kvq_decode_step: the decode step with each sequence's new token
quantized and written inside the decode call ("Output-Aware Rotation for INT2
KV-Cache Quantization", §6 cache-write kernel and decode; Eqs. 4, 20-22, 26, 27).

The fused step must write exactly the bytes kvq_quantize_append writes and return
exactly what kvq_decode_attention returns over the extended sequences (the same
warp slices, so bit for bit, also at a full wave where the two calls group the
warps into thread blocks differently), and both must match the fp64 oracle."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    # hq, hkv, page, lengths (after the step), rot, dtype, clips
    (8, 2, 16, [1, 16, 17, 300, 0, 33], "dense", "bf16", (0.96, 0.92)),
    (4, 4, 8, [9, 8, 1, 130], "signed_hadamard", "f32", (1.0, 0.9)),
    (32, 8, 16, [777, 2048], "dense", "bf16", (1.0, 1.0)),
    (8, 1, 16, [64, 65, 5], "identity", "bf16", (0.9, 0.9)),
    (40, 10, 16, [1100, 3000, 1025], "dense", "bf16", (1.0, 1.0)),
    # a full wave of the GPU (more than 16 chunks per warp of the default grid)
    (32, 8, 16, [3072] * 15 + [2900], "dense", "bf16", (0.96, 0.92)),
    # 8 query heads per KV head at a full wave: 12-warp blocks (6-warp blocks in the step)
    (64, 8, 16, [2048] * 15 + [1900], "signed_hadamard", "bf16", (1.0, 0.9)),
]


def _inputs(g):
    """History pools (every token but the last) and the step's new tokens."""
    c = g.case
    kv = [c.kv(b) for b in range(c.n_seqs)]
    hist = np.maximum(g.lengths - 1, 0)
    pool = g.new_pool()
    ks, vs, cu, start = [], [], [0], []
    for b in range(c.n_seqs):
        ks.append(kv[b][0][:hist[b]])
        vs.append(kv[b][1][:hist[b]])
        cu.append(cu[-1] + int(hist[b]))
        start.append(0)
    g.kvq.kvq_quantize_append(g.layout, gu.dev(np.concatenate(ks), c.dtype), gu.dev(np.concatenate(vs), c.dtype),
                              gu.dev_i32(cu), gu.dev_i32(start), g.table, g.rot_k, g.rot_v, g.mu_rot_dev, c.clip_k,
                              c.clip_v, pool)
    zero = np.zeros((c.n_kv_heads, 128), np.float32)
    k_new = np.stack([kv[b][0][g.lengths[b] - 1] if g.lengths[b] else zero for b in range(c.n_seqs)])
    v_new = np.stack([kv[b][1][g.lengths[b] - 1] if g.lengths[b] else zero for b in range(c.n_seqs)])
    return pool, k_new, v_new


@pytest.mark.parametrize("hq,hkv,page,lengths,rot,dtype,clips", CASES, ids=lambda v: str(v))
def test_step_equals_append_then_decode_and_the_oracle(hq, hkv, page, lengths, rot, dtype, clips):
    case = W.decode_case(61, lengths, hq, hkv, 128, rot, dtype, page_tokens=page, clip_k=clips[0], clip_v=clips[1],
                         spare_blocks=2, n_cal=256)
    g = gu.GpuCase(case)
    kvq, torch = g.kvq, g.torch
    pool_a, k_new, v_new = _inputs(g)
    pool_b = pool_a.clone()
    max_len = int(g.lengths.max())
    q = gu.dev(case.queries(), dtype)
    kn, vn = gu.dev(k_new, dtype), gu.dev(v_new, dtype)
    lens = gu.dev_i32(g.lengths)
    ws = torch.empty(max(kvq.kvq_decode_workspace_size(g.layout, case.n_seqs, max_len), 16), dtype=torch.uint8,
                     device="cuda")
    # separate calls: append the new tokens (sequences of length 0 append nothing), then decode
    has = g.lengths > 0
    kvq.kvq_quantize_append(g.layout, gu.dev(k_new[has], dtype), gu.dev(v_new[has], dtype),
                            gu.dev_i32(np.concatenate([[0], np.cumsum(has)])),
                            gu.dev_i32(np.maximum(g.lengths - 1, 0)), g.table, g.rot_k, g.rot_v, g.mu_rot_dev,
                            case.clip_k, case.clip_v, pool_a)
    out_a = torch.full((case.n_seqs, hq, 128), float("nan"), device="cuda")
    kvq.kvq_decode_attention(g.layout, q, lens, max_len, g.table, g.rot_k, pool_a, ws, out_a)
    # the fused step
    out_b = torch.full_like(out_a, float("nan"))
    kvq.kvq_decode_step(g.layout, q, kn, vn, lens, max_len, g.table, g.rot_k, g.rot_v, g.mu_rot_dev, case.clip_k,
                        case.clip_v, pool_b, ws, out_b)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(out_a, out_b)
    # and the oracle: pool bytes (with the boundary exemption) and the readout
    ora_pool, encs = g.oracle_pool()
    gu.compare_codes(pool_b.cpu().numpy(), ora_pool, hkv, page, case.block_table, g.lengths, encs,
                     (case.clip_k, case.clip_v), label="step")
    got = out_b.cpu().numpy()
    ref = g.oracle_decode(ora_pool, case.queries())
    for b in range(case.n_seqs):
        if g.lengths[b] == 0:
            assert np.all(got[b] == 0)
        else:
            assert gu.out_err(got[b], ref[b]) <= gu.OUT_TOL, (b, gu.out_err(got[b], ref[b]))


def test_consecutive_steps_walk_across_pages():
    """Twenty single-token steps on the same pool (lengths cross page boundaries):
    the pool ends byte-equal to the oracle's encoding of every token."""
    lengths0 = np.array([5, 30, 1, 250])
    n_steps = 20
    final = lengths0 + n_steps - 1
    case = W.decode_case(62, final, 8, 2, 128, "dense", "bf16", page_tokens=16, clip_k=0.96, clip_v=0.92, n_cal=256)
    g = gu.GpuCase(case, lengths=lengths0 - 1)
    kvq, torch = g.kvq, g.torch
    pool = g.new_pool()
    g.gpu_append_all(pool)  # history: lengths0 - 1 tokens
    kv = [case.kv(b) for b in range(case.n_seqs)]
    ws = torch.empty(kvq.kvq_decode_workspace_size(g.layout, case.n_seqs, int(final.max())), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(case.n_seqs, 8, 128, device="cuda")
    q = gu.dev(case.queries(), "bf16")
    for st in range(n_steps):
        lens = lengths0 + st
        k_new = np.stack([kv[b][0][lens[b] - 1] for b in range(case.n_seqs)])
        v_new = np.stack([kv[b][1][lens[b] - 1] for b in range(case.n_seqs)])
        kvq.kvq_decode_step(g.layout, q, gu.dev(k_new, "bf16"), gu.dev(v_new, "bf16"), gu.dev_i32(lens),
                            int(lens.max()), g.table, g.rot_k, g.rot_v, g.mu_rot_dev, case.clip_k, case.clip_v, pool,
                            ws, out)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    g.lengths = final
    ora_pool, encs = g.oracle_pool()
    gu.compare_codes(pool.cpu().numpy(), ora_pool, 2, 16, case.block_table, final, encs, (case.clip_k, case.clip_v),
                     label="steps")
    ref = g.oracle_decode(ora_pool, case.queries())
    got = out.cpu().numpy()
    for b in range(case.n_seqs):
        assert gu.out_err(got[b], ref[b]) <= gu.OUT_TOL


def _ties(rng, n, hkv):
    """Rotated groups on, next to and away from the code boundaries (min 0, max
    3 * step, the rest at k, k + 1/2 and k + 1/2 +- 2^-20 steps), [n][hkv][128]."""
    y = np.empty((n, hkv, 128))
    for i in range(n):
        for h in range(hkv):
            step = 2.0 ** rng.integers(-4, 2)
            k = rng.integers(0, 3, 128).astype(np.float64)
            kind = rng.integers(0, 4, 128)
            off = np.select([kind == 0, kind == 1, kind == 2],
                            [0.0, 0.5, 0.5 + 2.0 ** -20 * rng.choice([-1, 1], 128)], rng.uniform(0, 1, 128))
            v = (k + off) * step
            v[rng.integers(0, 64)] = 0.0
            v[64 + rng.integers(0, 64)] = 3.0 * step
            y[i, h] = np.clip(v, 0.0, 3.0 * step)
    return y


def test_step_with_several_sequences_per_query_block_and_near_ties():
    """384 (sequence, KV head) units: the query preparation appends for two sequences
    per block.  The new tokens are built so that their rotated, centred values sit on
    and next to the code boundaries (x = y R^T + mu with y on the grid, so x R is within
    fp32 rounding of a midpoint); their codes and fp16 meta must equal the fp64
    oracle's exactly, the rest of the pool and the readout as in the other cases."""
    import oracle
    rng = np.random.default_rng(65)
    lengths = rng.integers(20, 200, 48)
    case = W.decode_case(65, lengths, 32, 8, 128, "dense", "f32", page_tokens=16, clip_k=1.0, clip_v=1.0,
                         spare_blocks=2, n_cal=256)
    g = gu.GpuCase(case)
    mu = oracle.cache.key_mean(case.calibration_keys())
    yk, yv = _ties(rng, case.n_seqs, 8), _ties(rng, case.n_seqs, 8)
    orig = case.kv

    def kv(b):
        k, v = orig(b)
        k, v = k.copy(), v.copy()
        # y R^T per head (R orthogonal), so that (k - mu) R = y and v R = y up to fp32 rounding
        k[-1] = (np.einsum("hd,hcd->hc", yk[b], g.r_k) + mu).astype(np.float32)
        v[-1] = np.einsum("hd,hcd->hc", yv[b], g.r_v).astype(np.float32)
        return k, v

    case.kv = kv
    kvq, torch = g.kvq, g.torch
    pool, k_new, v_new = _inputs(g)
    max_len = int(g.lengths.max())
    q = gu.dev(case.queries(), "f32")
    ws = torch.empty(kvq.kvq_decode_workspace_size(g.layout, case.n_seqs, max_len), dtype=torch.uint8, device="cuda")
    out = torch.full((case.n_seqs, 32, 128), float("nan"), device="cuda")
    kvq.kvq_decode_step(g.layout, q, gu.dev(k_new, "f32"), gu.dev(v_new, "f32"), gu.dev_i32(g.lengths), max_len,
                        g.table, g.rot_k, g.rot_v, g.mu_rot_dev, case.clip_k, case.clip_v, pool, ws, out)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    ora_pool, encs = g.oracle_pool()
    gpool = pool.cpu().numpy()
    for b in range(case.n_seqs):
        n = int(g.lengths[b])
        for which in ("k", "v"):
            cg, mg = gu.seq_codes_meta(gpool, 8, 16, case.block_table[b], n, which)
            co, mo = gu.seq_codes_meta(ora_pool, 8, 16, case.block_table[b], n, which)
            assert np.array_equal(cg[-1], co[-1]), (b, which, int((cg[-1] != co[-1]).sum()))
            assert np.array_equal(mg[-1], mo[-1]), (b, which)
    gu.compare_codes(gpool, ora_pool, 8, 16, case.block_table, g.lengths, encs, (case.clip_k, case.clip_v),
                     label="step ties")
    got = out.cpu().numpy()
    ref = g.oracle_decode(ora_pool, case.queries())
    for b in range(case.n_seqs):
        assert gu.out_err(got[b], ref[b]) <= gu.OUT_TOL, (b, gu.out_err(got[b], ref[b]))


def test_step_and_projection_with_pinned_host_buffers():
    """The C-ABI takes plain pointers: q and the new K/V in pinned host memory (read by the
    query preparation over the host link) and y in pinned host memory (written by the
    projection) give the same pool, o_rot and y as device buffers, bit for bit."""
    lengths, hq, hkv, d_model = [700, 33, 1, 2048], 8, 2, 256
    case = W.decode_case(63, lengths, hq, hkv, d_model, "dense", "bf16", page_tokens=16, clip_k=0.96, clip_v=0.92,
                         spare_blocks=2, n_cal=256)
    g = gu.GpuCase(case)
    kvq, torch = g.kvq, g.torch
    pool_a, k_new, v_new = _inputs(g)
    pool_b = pool_a.clone()
    max_len = int(g.lengths.max())
    q_np = case.queries()
    q, kn, vn = gu.dev(q_np, "bf16"), gu.dev(k_new, "bf16"), gu.dev(v_new, "bf16")
    qh, knh, vnh = q.cpu().pin_memory(), kn.cpu().pin_memory(), vn.cpu().pin_memory()
    lens = gu.dev_i32(g.lengths)
    ws = torch.empty(max(kvq.kvq_decode_workspace_size(g.layout, case.n_seqs, max_len), 16), dtype=torch.uint8,
                     device="cuda")
    w = gu.dev(case.w_o(), "bf16")
    wp = torch.empty(kvq.kvq_wo_packed_bytes(d_model, hq * 128), dtype=torch.uint8, device="cuda")
    kvq.kvq_pack_wo(w, wp)
    o_a = torch.full((case.n_seqs, hq, 128), float("nan"), device="cuda")
    y_a = torch.full((case.n_seqs, d_model), float("nan"), device="cuda")
    kvq.kvq_decode_step(g.layout, q, kn, vn, lens, max_len, g.table, g.rot_k, g.rot_v, g.mu_rot_dev, case.clip_k,
                        case.clip_v, pool_a, ws, o_a)
    kvq.kvq_out_proj_packed(o_a.reshape(case.n_seqs, -1), wp, y_a, d_model)
    o_b = torch.full_like(o_a, float("nan"))
    y_b = torch.full((case.n_seqs, d_model), float("nan")).pin_memory()
    kvq.kvq_decode_step(g.layout, qh, knh, vnh, lens, max_len, g.table, g.rot_k, g.rot_v, g.mu_rot_dev, case.clip_k,
                        case.clip_v, pool_b, ws, o_b)
    kvq.kvq_out_proj_packed(o_b.reshape(case.n_seqs, -1), wp, y_b, d_model)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(o_a, o_b)
    assert torch.equal(y_a.cpu(), y_b)
    # the decode alone with the query in host memory
    o_c, o_d = torch.full_like(o_a, float("nan")), torch.full_like(o_a, float("nan"))
    kvq.kvq_decode_attention(g.layout, q, lens, max_len, g.table, g.rot_k, pool_a, ws, o_c)
    kvq.kvq_decode_attention(g.layout, qh, lens, max_len, g.table, g.rot_k, pool_a, ws, o_d)
    torch.cuda.synchronize()
    assert torch.equal(o_c, o_d)
