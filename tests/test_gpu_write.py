"""GPU parity of the write path: kvq_quantize_append, kvq_key_mean, kvq_rotate_heads."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    # rot, dtype, page, lengths, clips
    ("identity", "f32", 16, [1, 37, 300], (1.0, 1.0)),
    ("signed_hadamard", "f32", 16, [16, 129, 5], (0.9, 0.95)),
    ("signed_hadamard", "bf16", 8, [300, 17], (1.0, 0.85)),
    ("dense", "f32", 8, [33, 250], (0.96, 0.92)),
    ("dense", "bf16", 16, [511, 2, 64], (1.0, 1.0)),
    ("identity", "bf16", 8, [7, 8, 9], (0.8, 0.8)),
    # at most 128 new tokens per call with dense R: the decode-step kernel (certified fp32, double-float redo)
    ("dense", "bf16", 16, [1, 37, 60], (0.95, 0.9)),
    ("dense", "f32", 8, [5, 3, 9], (1.0, 0.85)),
]


@pytest.mark.parametrize("rot,dtype,page,lengths,clips", CASES, ids=lambda v: str(v))
def test_quantize_append_matches_oracle(rot, dtype, page, lengths, clips):
    case = W.decode_case(11, lengths, 4, 2, 256, rot, dtype, page_tokens=page, clip_k=clips[0], clip_v=clips[1],
                         spare_blocks=3, n_cal=256)
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    g.kvq.kvq_device_check()
    ora_pool, encs = g.oracle_pool()
    gpool = pool.cpu().numpy()
    stats = gu.compare_codes(gpool, ora_pool, case.n_kv_heads, page, case.block_table, g.lengths, encs,
                             (case.clip_k, case.clip_v),
                             label=f"{rot}/{dtype}/P{page}")
    # bytes of pages that no sequence owns stay untouched (zero) on both sides
    used = np.zeros(case.num_blocks, bool)
    for b, n in enumerate(g.lengths):
        used[case.block_table[b, :(n + page - 1) // page]] = True
    rec = gpool.reshape(case.num_blocks, -1)
    assert rec[~used].sum() == 0
    print("code parity", stats)


@pytest.mark.parametrize("rot,chunks", [("signed_hadamard", 3), ("dense", 3), ("dense", 8)])
def test_chunked_append_equals_single_append(rot, chunks):
    # chunks=8 puts <= 128 tokens in each call: the decode-step kernel (certified fp32 with a
    # double-float redo) against the double-float shared-R kernel of the single call: equal codes
    case = W.decode_case(12, [300, 45, 160], 8, 4, 128, rot, "bf16", page_tokens=16, clip_k=0.9, n_cal=128)
    g = gu.GpuCase(case)
    a = g.new_pool()
    b = g.new_pool()
    g.gpu_append_all(a, chunks=1)
    g.gpu_append_all(b, chunks=chunks)  # chunk edges fall inside pages
    assert g.torch.equal(a, b)


def test_identity_rotation_equals_plain_int2_on_gpu():
    # pin: the identity rotation is plain INT2 (Eq. 4 with R = I); uncentred, clip 1
    case = W.decode_case(13, [100], 1, 1, 128, "identity", "f32", n_off=0)
    g = gu.GpuCase(case, mu_mode="none")
    pool = g.new_pool()
    g.gpu_append_all(pool)
    import oracle
    k, v = case.kv(0)
    codes, s, z = oracle.quant.quantize_groups(k.astype(np.float64), 1.0)
    ck, mk = gu.seq_codes_meta(pool.cpu().numpy(), 1, 16, case.block_table[0], 100, "k")
    assert np.array_equal(ck, codes)
    assert np.array_equal(mk[..., 0], oracle.quant.fp16_bits(s)) and np.array_equal(mk[..., 1], oracle.quant.fp16_bits(z))


@pytest.mark.parametrize("rot,n_tok", [("signed_hadamard", 40), ("dense", 300)])
def test_out_of_range_block_is_skipped_and_flagged(rot, n_tok):
    # dense with 300 tokens: the tensor-core cache write locates the tokens of its tiles
    case = W.decode_case(14, [n_tok], 2, 2, 128, rot, "f32", page_tokens=16, spare_blocks=1)
    case.block_table[0, 1] = case.num_blocks + 5  # page 1 points outside the pool
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    with pytest.raises(g.kvq.KvqError) as e:
        g.kvq.kvq_device_check()
    assert e.value.status == g.kvq.KVQ_EDEVICE_FLAG
    g.kvq.kvq_device_check()  # the word was cleared
    # pages 0 and 2 were written, nothing else
    rec = pool.cpu().numpy().reshape(case.num_blocks, -1)
    assert rec[case.block_table[0, 0]].any() and rec[case.block_table[0, 2]].any()


def test_key_mean_and_rotate_heads_match_oracle():
    import oracle
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    case = W.decode_case(15, [8], 8, 4, 128, "dense", "bf16", n_cal=1000)
    kc = case.calibration_keys()
    mu = torch.empty(4, 128, device="cuda")
    kvq.kvq_key_mean(gu.dev(kc, "bf16"), mu)
    ref = oracle.cache.key_mean(kc)
    assert np.abs(mu.cpu().numpy() - ref).max() <= 1e-6 * np.abs(ref).max()
    for rot in ("identity", "signed_hadamard", "dense"):
        spec = W.make_rot(rot, 15, 3, 4)
        r = oracle.rotations.rot_matrices(spec, 4)
        x = np.random.default_rng(0).standard_normal((5, 8, 128)).astype(np.float32)
        y = torch.empty(5, 8, 128, device="cuda")
        kvq.kvq_rotate_heads(gu.dev(x), kvq.DeviceRot.from_spec(spec), y, heads_per_rot=2)
        yr = oracle.cache.rotate_heads(x, r, heads_per_rot=2)
        assert gu.normwise_err(y.cpu().numpy(), yr) < 1e-6, rot


def _tie_groups(rng, n_tok, n_heads):
    """Groups whose exact values sit on, next to and away from the code
    boundaries: min 0 and max 3 * step (so scale = step, zero = 0 exactly), the
    rest at k * step, (k + 1/2) * step (exact ties), (k + 1/2) * step +- step *
    2^-23 (inside the fp32 decision's error bound) and +- step * 2^-14 (outside)."""
    x = np.empty((n_tok, n_heads, 128), np.float32)
    for t in range(n_tok):
        for h in range(n_heads):
            step = np.float32(2.0 ** rng.integers(-6, 4))
            k = rng.integers(0, 3, 128).astype(np.float64)
            kind = rng.integers(0, 5, 128)
            off = np.select([kind == 0, kind == 1, kind == 2, kind == 3],
                            [0.0, 0.5, 0.5 + 2.0 ** -23 * rng.choice([-1, 1], 128),
                             0.5 + 2.0 ** -14 * rng.choice([-1, 1], 128)], rng.uniform(0, 1, 128))
            v = (k + off) * step
            v[rng.integers(0, 64)] = 0.0
            v[64 + rng.integers(0, 64)] = 3.0 * step
            x[t, h] = np.clip(v, 0.0, 3.0 * step).astype(np.float32)
    return x


def test_exact_ties_and_near_ties_match_the_oracle():
    """Codes on and next to the rounding midpoints (identity rotation, fp32 input,
    no centring) equal the fp64 oracle's: the certified fp32 decision must hand
    every uncertain group to the double-float path, which breaks ties to even."""
    import oracle
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    rng = np.random.default_rng(2718)
    n_tok, hkv, page = 160, 2, 16
    k = _tie_groups(rng, n_tok, hkv)
    v = _tie_groups(rng, n_tok, hkv)
    nb = n_tok // page
    lay = kvq.make_layout(page, hkv, hkv, nb, nb)
    pool = torch.zeros(kvq.kvq_pool_bytes(lay), dtype=torch.uint8, device="cuda")
    ident = kvq.DeviceRot("identity")
    kvq.kvq_quantize_append(lay, gu.dev(k), gu.dev(v), gu.dev_i32([0, n_tok]), gu.dev_i32([0]),
                            gu.dev_i32(np.arange(nb)[None, :]), ident, ident, None, 1.0, 1.0, pool)
    kvq.kvq_device_check()
    gpool = pool.cpu().numpy()
    for which, x in (("k", k), ("v", v)):
        codes, s, z = oracle.quant.quantize_groups(x.astype(np.float64), 1.0)
        got_c, got_m = gu.seq_codes_meta(gpool, hkv, page, np.arange(nb), n_tok, which)
        assert np.array_equal(got_m[..., 0], oracle.quant.fp16_bits(s)), which
        assert np.array_equal(got_m[..., 1], oracle.quant.fp16_bits(z)), which
        assert np.array_equal(got_c, codes), (which, int((got_c != codes).sum()))


def _signed_permutations(rng, n_heads):
    """Dense R that are signed permutation matrices: x R is exact in any arithmetic."""
    r = np.zeros((n_heads, 128, 128), np.float32)
    for h in range(n_heads):
        r[h, np.arange(128), rng.permutation(128)] = rng.choice([-1.0, 1.0], 128)
    return r


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dense_bulk_append_exact_on_ties(dtype):
    """More than 128 new tokens with dense R: the tensor-core cache write.  With
    signed-permutation R the rotated values are exact, and the groups sit on and
    next to the code and fp16 rounding boundaries, so most groups leave the fp32
    decision uncertain: scale, zero and codes then come from double-float values
    of the uncertain elements and must equal the fp64 oracle's bit for bit (ties
    to even).  300 tokens: two full tiles and a ragged one."""
    import oracle
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    rng = np.random.default_rng(3141)
    n_tok, hkv, page = 300, 2, 16
    k = _tie_groups(rng, n_tok, hkv)
    v = _tie_groups(rng, n_tok, hkv)
    if dtype == "bf16":
        k, v = W.round_bf16(k), W.round_bf16(v)
    rk, rv = _signed_permutations(rng, hkv), _signed_permutations(rng, hkv)
    nb = (n_tok + page - 1) // page
    lay = kvq.make_layout(page, hkv, hkv, nb, nb)
    pool = torch.zeros(kvq.kvq_pool_bytes(lay), dtype=torch.uint8, device="cuda")
    dk = kvq.DeviceRot("dense", dense=gu.dev(rk))
    dv = kvq.DeviceRot("dense", dense=gu.dev(rv))
    kvq.kvq_quantize_append(lay, gu.dev(k, dtype), gu.dev(v, dtype), gu.dev_i32([0, n_tok]), gu.dev_i32([0]),
                            gu.dev_i32(np.arange(nb)[None, :]), dk, dv, None, 1.0, 0.9, pool)
    kvq.kvq_device_check()
    gpool = pool.cpu().numpy()
    for which, x, r, clip in (("k", k, rk, 1.0), ("v", v, rv, 0.9)):
        y = np.einsum("thc,hcd->thd", x.astype(np.float64), r.astype(np.float64))
        codes, s, z = oracle.quant.quantize_groups(y, clip)
        got_c, got_m = gu.seq_codes_meta(gpool, hkv, page, np.arange(nb), n_tok, which)
        assert np.array_equal(got_m[..., 0], oracle.quant.fp16_bits(s)), which
        assert np.array_equal(got_m[..., 1], oracle.quant.fp16_bits(z)), which
        assert np.array_equal(got_c, codes), (which, int((got_c != codes).sum()))


def test_dense_keys_hadamard_values_bulk_append():
    """Dense R_K with signed-Hadamard R_V in one call of more than 128 tokens: the
    tensor-core kernel takes the keys alone, the Walsh-Hadamard kernel the values."""
    case = W.decode_case(16, [200, 97], 4, 2, 256, "dense", "bf16", page_tokens=8, clip_k=0.95, clip_v=0.9,
                         spare_blocks=2, n_cal=256)
    case.rot_v = W.make_rot("signed_hadamard", 16, 7, case.n_kv_heads)
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    g.kvq.kvq_device_check()
    ora_pool, encs = g.oracle_pool()
    stats = gu.compare_codes(pool.cpu().numpy(), ora_pool, case.n_kv_heads, 8, case.block_table, g.lengths, encs,
                             (case.clip_k, case.clip_v), label="dense K / Hadamard V")
    assert stats["mismatch"] == 0 and stats["meta_mismatch_groups"] == 0, stats


@pytest.mark.parametrize("dtype,lengths", [("f32", [5000, 4999]), ("bf16", [3000, 2900, 3100])])
def test_dense_bulk_append_many_units_per_cta(dtype, lengths):
    """More (role, head, 128-token tile) units than SMs: every persistent CTA of the
    tensor-core cache write takes several units, restages R when the head changes and
    (bf16) copies the next tile's rows while the current one is decided; codes and meta
    equal the oracle's."""
    case = W.decode_case(17, lengths, 8, 4, 256, "dense", dtype, page_tokens=16, clip_k=0.9, clip_v=0.96,
                         spare_blocks=2, n_cal=256)
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    g.kvq.kvq_device_check()
    ora_pool, encs = g.oracle_pool()
    stats = gu.compare_codes(pool.cpu().numpy(), ora_pool, case.n_kv_heads, 16, case.block_table, g.lengths, encs,
                             (case.clip_k, case.clip_v), label=f"dense {dtype} many units")
    assert stats["mismatch"] == 0 and stats["meta_mismatch_groups"] == 0, stats
