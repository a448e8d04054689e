"""GPU parity of kvq_fold_wo and kvq_out_proj against the fp64 oracle."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rot,wdt,odt", [("dense", "bf16", "f32"), ("signed_hadamard", "f32", "f32"),
                                         ("dense", "bf16", "bf16"), ("identity", "f32", "bf16")])
def test_fold_wo(rot, wdt, odt):
    import oracle
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    hq, hkv, dm = 8, 2, 320
    w = W.draw_wo(31, dm, hq * 128, wdt)
    spec = W.make_rot(rot, 31, 1, hkv)
    r = oracle.rotations.rot_matrices(spec, hkv)
    out = torch.empty(dm, hq * 128, device="cuda", dtype=torch.float32 if odt == "f32" else torch.bfloat16)
    kvq.kvq_fold_wo(gu.dev(w, wdt), hq, hkv, kvq.DeviceRot.from_spec(spec), out)
    ref = oracle.output.fold_wo(w, r, hq // hkv)
    got = out.float().cpu().numpy()
    if odt == "f32":
        assert gu.normwise_err(got, ref) < 1e-6
    else:
        # bf16 output: within one bf16 rounding of the exact fold
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("rows,dm,hq,wdt", [(1, 128, 1, "f32"), (16, 4096, 32, "bf16"), (5, 200, 3, "bf16"),
                                            (64, 640, 10, "f32"), (48, 520, 5, "bf16"), (64, 5120, 40, "bf16"),
                                            (100, 256, 2, "bf16"), (27, 3300, 3, "bf16"),
                                            # cluster sizes (K split) 5 and 8, one and two 8-row groups:
                                            (8, 3328, 8, "bf16"), (11, 3300, 8, "bf16"), (9, 3300, 3, "bf16")])
def test_out_proj(rows, dm, hq, wdt):
    import oracle
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    w = W.draw_wo(32, dm, hq * 128, wdt)
    o = np.random.default_rng(1).standard_normal((rows, hq, 128)).astype(np.float32)
    y = torch.empty(rows, dm, device="cuda")
    kvq.kvq_out_proj(gu.dev(o).reshape(rows, -1), gu.dev(w, wdt), y)
    ref = oracle.output.out_proj(o, w)
    assert gu.out_err(y.cpu().numpy(), ref) <= gu.OUT_TOL


def test_folded_projection_of_rotated_readout_equals_unrotated():
    """Eq. 31 on the GPU: out_proj(o R_V, fold(W_O)) = o W_O^T."""
    import oracle
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    hq, hkv, dm = 8, 4, 256
    w = W.draw_wo(33, dm, hq * 128, "f32")
    spec = W.make_rot("dense", 33, 2, hkv)
    r = oracle.rotations.rot_matrices(spec, hkv)
    o = np.random.default_rng(2).standard_normal((3, hq, 128))
    o_rot = np.einsum("bjc,jcd->bjd", o, r[np.arange(hq) // 2]).astype(np.float32)
    wf = torch.empty(dm, hq * 128, device="cuda")
    kvq.kvq_fold_wo(gu.dev(w), hq, hkv, kvq.DeviceRot.from_spec(spec), wf)
    y = torch.empty(3, dm, device="cuda")
    kvq.kvq_out_proj(gu.dev(o_rot).reshape(3, -1), wf, y)
    assert gu.normwise_err(y.cpu().numpy(), oracle.output.out_proj(o, w)) < 1e-4


@pytest.mark.parametrize("rows,dm,k", [(70, 300, 96), (1, 129, 32), (64, 1000, 160), (65, 256, 4096)])
def test_out_proj_ragged_k_and_passes(rows, dm, k):
    """K not a multiple of the 64-column stage (the last stage reads zeros past the edge),
    d_model not a multiple of the 128-row tile, and row counts around the 64-row pass."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    rng = np.random.default_rng(rows * 7 + k)
    w = (rng.standard_normal((dm, k)) / np.sqrt(k)).astype(np.float32)
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()  # bf16-exact weights
    x = rng.standard_normal((rows, k)).astype(np.float32)
    y = torch.empty(rows, dm, device="cuda")
    kvq.kvq_out_proj(gu.dev(x), gu.dev(w, "bf16"), y)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert gu.out_err(y.cpu().numpy(), ref) <= gu.OUT_TOL


def _unpack(packed, d_model, k_dim):
    """Read the packed W back (the documented box order) as a [d_model][k_dim] bf16-bit array."""
    n_kb = (k_dim + 63) // 64
    n_mt = (d_model + 127) // 128
    b = packed.reshape(n_mt, n_kb, 128, 8, 8)  # [tile][stage][row][chunk position][8 bf16 bits]
    out = np.zeros((n_mt * 128, n_kb * 64), np.uint16)
    r = np.arange(128)
    for jj in range(8):
        j = jj ^ (r & 7)  # the source chunk stored at position jj of row r
        for T in range(n_mt):
            for c in range(n_kb):
                for rr in range(128):
                    out[T * 128 + rr, c * 64 + 8 * j[rr]:c * 64 + 8 * j[rr] + 8] = b[T, c, rr, jj]
    return out[:d_model, :k_dim]


@pytest.mark.parametrize("n_rows,d_model,k_dim", [(16, 4096, 4096), (64, 5120, 5120), (3, 300, 4096), (9, 256, 160),
                                                  (1, 128, 32)])
def test_packed_projection_equals_row_major(n_rows, d_model, k_dim):
    """kvq_pack_wo's box order read back equals W bit for bit, and kvq_out_proj_packed returns
    exactly what kvq_out_proj returns with the row-major bf16 W (same products, same order)."""
    torch = gu.torch_cuda()
    kvq = gu.kvq_lib()
    gen = np.random.default_rng(d_model + k_dim)
    w = torch.from_numpy(gen.standard_normal((d_model, k_dim)).astype(np.float32) / np.sqrt(k_dim)).cuda()
    w = w.to(torch.bfloat16)
    x = torch.from_numpy(gen.standard_normal((n_rows, k_dim)).astype(np.float32)).cuda()
    packed = torch.full((kvq.kvq_wo_packed_bytes(d_model, k_dim),), 0x5A, dtype=torch.uint8, device="cuda")
    kvq.kvq_pack_wo(w, packed)
    y_rm = torch.empty(n_rows, d_model, device="cuda")
    y_pk = torch.full_like(y_rm, float("nan"))
    kvq.kvq_out_proj(x, w, y_rm)
    kvq.kvq_out_proj_packed(x, packed, y_pk, d_model)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    if d_model * k_dim <= 300 * 4096:
        got = _unpack(packed.cpu().numpy().view(np.uint16), d_model, k_dim)
        assert np.array_equal(got, w.view(torch.int16).cpu().numpy().view(np.uint16))
    assert torch.equal(y_pk, y_rm)
