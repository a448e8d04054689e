"""GPU parity of the read path: kvq_decode_attention against the fp64 oracle.

The GPU decodes the pool written by the oracle (so both sides read identical
codes), and separately its own pool end to end."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    # hq, hkv, page, lengths, rot, dtype, splits
    (1, 1, 16, [512], "signed_hadamard", "f32", 0),
    (4, 1, 16, [1, 15, 16, 17, 300], "dense", "f32", 0),
    (8, 2, 8, [257, 64, 3], "identity", "bf16", 3),
    (32, 4, 16, [1000, 0, 777], "signed_hadamard", "bf16", 0),
    (16, 2, 16, [2049, 600], "dense", "bf16", 7),
    (16, 16, 8, [100, 90], "dense", "f32", 1),
]


@pytest.mark.parametrize("hq,hkv,page,lengths,rot,dtype,splits", CASES, ids=lambda v: str(v))
def test_decode_on_oracle_pool(hq, hkv, page, lengths, rot, dtype, splits):
    case = W.decode_case(21, lengths, hq, hkv, 128, rot, dtype, page_tokens=page, clip_k=0.95, n_cal=256)
    g = gu.GpuCase(case)
    ora_pool, _ = g.oracle_pool()
    pool = g.torch.from_numpy(ora_pool).cuda()
    q = case.queries()
    got = g.gpu_decode(pool, q, n_splits=splits)
    g.kvq.kvq_device_check()
    ref = g.oracle_decode(ora_pool, q)
    for b in range(case.n_seqs):
        err = gu.out_err(got[b], ref[b]) if np.abs(ref[b]).max() > 0 else np.abs(got[b]).max()
        assert err <= gu.OUT_TOL, (b, err)
        assert np.isfinite(got[b]).all()
    assert np.all(got[np.asarray(lengths) == 0] == 0)


@pytest.mark.parametrize("splits", [1, 2, 5, 64])
def test_split_count_does_not_change_the_result(splits):
    case = W.decode_case(22, [3000, 1234], 8, 2, 128, "signed_hadamard", "bf16", n_cal=128)
    g = gu.GpuCase(case)
    ora_pool, _ = g.oracle_pool()
    pool = g.torch.from_numpy(ora_pool).cuda()
    q = case.queries()
    ref = g.gpu_decode(pool, q, n_splits=1)
    got = g.gpu_decode(pool, q, n_splits=splits)
    # Split counts change only the order of fp32 (and tensor-core) accumulation;
    # the results agree ~40x inside the 2e-3 output tolerance.
    assert gu.normwise_err(got, ref) < 5e-5


def test_end_to_end_gpu_write_then_gpu_decode():
    case = W.decode_case(23, [700, 130], 16, 4, 128, "dense", "bf16", clip_k=0.96, clip_v=0.92, n_cal=256)
    g = gu.GpuCase(case)
    pool = g.new_pool()
    g.gpu_append_all(pool)
    q = case.queries()
    got = g.gpu_decode(pool, q)
    ora_pool, _ = g.oracle_pool()
    ref = g.oracle_decode(ora_pool, q)
    for b in range(case.n_seqs):
        assert gu.out_err(got[b], ref[b]) <= gu.OUT_TOL


def test_bad_sequence_length_is_flagged():
    case = W.decode_case(24, [40, 40], 2, 2, 128, "identity", "f32")
    g = gu.GpuCase(case)
    ora_pool, _ = g.oracle_pool()
    pool = g.torch.from_numpy(ora_pool).cuda()
    g.lengths = np.array([40, 10_000])  # beyond the block table
    with pytest.raises(g.kvq.KvqError):
        g.gpu_decode(pool, case.queries())  # max_seq_len check on the host
    # device-side check: max_seq_len within bounds, but one length negative
    kvq = g.kvq
    ws = g.torch.empty(kvq.kvq_decode_workspace_size(g.layout, 2, 40, 1), dtype=g.torch.uint8, device="cuda")
    out = g.torch.empty(2, 2, 128, device="cuda")
    kvq.kvq_decode_attention(g.layout, gu.dev(case.queries()), gu.dev_i32([40, -3]), 40, g.table, g.rot_k, pool,
                             ws, out, n_splits=1)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_device_check()
    assert e.value.status == kvq.KVQ_EDEVICE_FLAG
