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


def test_report_at_the_serving_calibration_size():
    """The size `bench.py --case report` runs: the 14B-class calibration trace (2,560
    tokens, the last 64 positions, 10 KV heads x 4 query heads, d_model 5,120, bf16), two
    dense candidates as R_K and R_V, centring, Table A's clips.  The GPU reports all ten
    heads; the oracle recomputes heads 0 and 9 from their slices of the inputs."""
    import oracle
    cc = W.serve14b_calibration(n_cand=2)
    mu = oracle.cache.key_mean(cc.k).astype(np.float32)
    rot_k, rot_v = cc.cands[:2]
    clips = (W.f32(0.96), W.f32(0.92))
    got = run_report(cc, rot_k, rot_v, mu, *clips)
    assert np.isfinite(got).all()
    r_k = oracle.rotations.rot_matrices(rot_k, cc.n_kv_heads)
    r_v = oracle.rotations.rot_matrices(rot_v, cc.n_kv_heads)
    g, D = cc.gqa, 128
    for h in (0, 9):
        qh = cc.q[:, h * g:(h + 1) * g]
        wh = cc.w_o[:, h * g * D:(h + 1) * g * D]
        rep = oracle.report.head_error_report(qh, cc.k[:, h:h + 1], cc.v[:, h:h + 1], wh, r_k[h:h + 1],
                                              r_v[h:h + 1], mu[h:h + 1], clips[0], clips[1], g)
        for i, name in enumerate(("e", "e_key", "e_val", "e_naive", "y")):
            gu.assert_nmse_close(got[i][h:h + 1], rep[name], f"head {h} {name}")
