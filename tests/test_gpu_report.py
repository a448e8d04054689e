"""GPU parity of kvq_head_error_report (per-head output error, Eq. 8 split)
against the fp64 oracle."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_report(cc, rk, rv, mu, clip_k, clip_v):
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    hkv, gqa = cc.n_kv_heads, cc.gqa
    ws = torch.empty(kvq.kvq_report_workspace_size(cc.n_tok, cc.n_qpos, hkv, gqa), dtype=torch.uint8, device="cuda")
    out = torch.full((5, hkv), float("nan"), dtype=torch.float64, device="cuda")
    kvq.kvq_head_error_report(gu.dev(cc.q, cc.dtype), gu.dev(cc.k, cc.dtype), gu.dev(cc.v, cc.dtype),
                              gu.dev(cc.w_o, cc.dtype), kvq.DeviceRot.from_spec(rk), kvq.DeviceRot.from_spec(rv),
                              gu.dev(mu) if mu is not None else None, clip_k, clip_v, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


CASES = [
    # seed, n_tok, n_qpos, hkv, gqa, d_model, rot_k, rot_v, centred, clips, dtype
    (51, 300, 7, 2, 4, 256, "dense", "dense", True, (0.96, 0.92), "f32"),
    (52, 200, 5, 2, 2, 96, "signed_hadamard", "dense", False, (1.0, 1.0), "f32"),   # d_model <= 128: direct form
    (53, 257, 9, 1, 8, 512, "dense", "signed_hadamard", True, (0.9, 0.9), "bf16"),
    (54, 130, 3, 4, 1, 300, "identity", "identity", False, (0.95, 0.95), "f32"),  # the plain INT2 itself
]


@pytest.mark.parametrize("seed,n_tok,n_qpos,hkv,gqa,d_model,rk,rv,centred,clips,dtype", CASES, ids=lambda v: str(v))
def test_report_matches_the_oracle(seed, n_tok, n_qpos, hkv, gqa, d_model, rk, rv, centred, clips, dtype):
    import oracle
    cc = W.small_calibration(seed, n_tok, n_qpos, hkv, gqa, d_model, kinds=(rk, rv), dtype=dtype)
    mu = oracle.cache.key_mean(cc.k).astype(np.float32) if centred else None
    rot_k, rot_v = cc.cands
    got = run_report(cc, rot_k, rot_v, mu, *clips)
    rep = oracle.report.head_error_report(cc.q, cc.k, cc.v, cc.w_o, oracle.rotations.rot_matrices(rot_k, hkv),
                                          oracle.rotations.rot_matrices(rot_v, hkv), mu,
                                          float(np.float32(clips[0])), float(np.float32(clips[1])), gqa)
    for i, name in enumerate(("e", "e_key", "e_val", "e_naive", "y")):
        gu.assert_nmse_close(got[i], rep[name], name)
    if rk == rv == "identity" and not centred:
        assert np.array_equal(got[0], got[3])  # the candidate is the plain INT2: identical passes
    pct = 100 * np.sqrt(got[0] / got[3])
    assert np.allclose(pct, rep["rms_pct_of_naive"], rtol=1e-4)
