"""kvq_decode_attention_noalloc: decode attention for callers that may not
allocate device memory (engines that reserve all memory up front and forbid
allocation while serving, plugin hosts that only hand over tensors).

The entry point keeps its split partials in a fixed buffer inside the library.
Here it is called through the C ABI twice in a row and must agree with the
ordinary entry point (which uses a caller-provided workspace) within the
attention tolerance, and a request too large for its buffer must be refused
with a clear error.  The file sorts last so that a run stopping at the first
failure has already run every other test; it depends on nothing those tests
leave behind.
"""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode_twice():
    case = W.decode_case(91, [777, 64, 2048, 1], 16, 4, 128, "dense", "bf16", clip_k=0.96, clip_v=0.92, n_cal=256)
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    kvq, torch = g.kvq, g.torch
    q = gu.dev(case.queries(), "bf16")
    lens = gu.dev_i32(case.seq_lens)
    max_len = int(case.seq_lens.max())
    ws = torch.empty(kvq.kvq_decode_workspace_size(g.layout, case.n_seqs, max_len), dtype=torch.uint8, device="cuda")
    ref = torch.empty(case.n_seqs, case.n_q_heads, 128, device="cuda")
    kvq.kvq_decode_attention(g.layout, q, lens, max_len, g.table, g.rot_k, pool, ws, ref)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_decode_attention_noalloc(g.layout, q, lens, max_len, g.table, g.rot_k, pool, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert gu.out_err(out.cpu().numpy(), ref.cpu().numpy()) <= gu.OUT_TOL
    kvq.kvq_device_check()


def _largest_fitting_splits(kvq, layout, n_seqs, max_len, limit):
    """Brute force over the workspace sizes: the largest partition count below the
    library's default whose workspace fits in `limit` bytes."""
    auto = kvq.kvq_decode_workspace_size(layout, n_seqs, max_len, 0)
    assert auto > limit
    best = 0
    n = 1
    while True:
        b = kvq.kvq_decode_workspace_size(layout, n_seqs, max_len, n)
        if b >= auto:
            break
        if b <= limit:
            best = n
        n += 1
    return best


def test_noalloc_takes_the_largest_partition_count_that_fits():
    """The 8B-class GQA shape (16 sequences, 8 KV heads, 32 query heads, dense R) at
    4,096 tokens: the library's default grid needs more partials than the built-in
    4 MiB buffer holds, so the entry point runs with the largest partition count that
    fits.  The decode is deterministic for a given count, so its output equals the
    ordinary entry point's at that count bit for bit, on two calls in a row."""
    case = W.decode_case(92, [4096] * 16, 32, 8, 4096, "dense", "bf16", n_cal=256)
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    kvq, torch = g.kvq, g.torch
    q = gu.dev(case.queries(), "bf16")
    lens = gu.dev_i32(case.seq_lens)
    max_len = int(case.seq_lens.max())
    n = _largest_fitting_splits(kvq, g.layout, case.n_seqs, max_len, 4 << 20)
    assert n > 1
    ws = torch.empty(kvq.kvq_decode_workspace_size(g.layout, case.n_seqs, max_len, n), dtype=torch.uint8,
                     device="cuda")
    ref = torch.empty(case.n_seqs, case.n_q_heads, 128, device="cuda")
    kvq.kvq_decode_attention(g.layout, q, lens, max_len, g.table, g.rot_k, pool, ws, ref, n_splits=n)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_decode_attention_noalloc(g.layout, q, lens, max_len, g.table, g.rot_k, pool, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    kvq.kvq_device_check()


def test_noalloc_rejects_partials_larger_than_its_buffer():
    kvq = gu.kvq_lib()
    torch = gu.torch_cuda()
    # 2048 sequences x 64 query heads x 64 splits of partials is far beyond 4 MiB
    lay = kvq.make_layout(16, 8, 64, 16, 8)
    q = torch.zeros(2048, 64, 128, device="cuda")
    lens = torch.zeros(2048, dtype=torch.int32, device="cuda")
    table = torch.zeros(2048, 8, dtype=torch.int32, device="cuda")
    pool = torch.zeros(kvq.kvq_pool_bytes(lay), dtype=torch.uint8, device="cuda")
    out = torch.empty(2048, 64, 128, device="cuda")
    rot = kvq.DeviceRot("identity")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attention_noalloc(lay, q, lens, 128, table, rot, pool, out, n_splits=64)
    assert e.value.status == kvq.KVQ_EUNSUPPORTED
    assert "built-in scratch" in str(e.value)
