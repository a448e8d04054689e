"""GPU parity of the OptR gradient calibration (Algorithm 1 of "Output-Aware
Rotation for INT2 KV-Cache Quantization"; §4.2-4.5 Eqs. 11-18) against the fp64
oracle: the key and value objectives and their gradients with respect to the
generator, and whole calibration runs (Adam, selection on a held-out trace)."""
import numpy as np
import pytest

import gpu_util as gu
from int2_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

D = 128


def _dev64(x):
    torch = gu.torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).cuda()


def _dev32(x):
    torch = gu.torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _setup(c):
    q, k, v = c.train
    mu = k.mean(axis=0).astype(np.float32)
    return q, k, v, mu


def _gpu_loss_grad(kvq, phase, q, k, v, w, mu, r0, a, r_sel, clip_k, clip_v, lam):
    torch = gu.torch_cuda()
    ws = torch.empty(kvq.kvq_optr_workspace_size(k.shape[0], q.shape[0], q.shape[1]), dtype=torch.uint8,
                     device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    grad = torch.zeros(D, D, dtype=torch.float64, device="cuda")
    kvq.kvq_optr_loss_grad(phase, _dev32(q), _dev32(k), _dev32(v), _dev32(w), _dev32(mu), _dev64(r0), _dev64(a),
                           _dev64(r_sel) if r_sel is not None else None, clip_k, clip_v, lam, loss, grad, ws)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    return float(loss.cpu().numpy()[0]), grad.cpu().numpy()


# clip ratios, lambda_K and the learning rate cross the ABI as float32: the oracle gets the same values
F32 = W.f32


@pytest.mark.parametrize("n_tok,n_qpos,gqa,d_model,clips,lam", [
    (48, 6, 2, 16, (0.96, 0.92), 1.0),
    (130, 9, 4, 300, (1.0, 0.9), 0.7),
    (64, 64, 1, 128, (0.9, 1.0), 1.0),
])
def test_losses_and_gradients_match_the_oracle(n_tok, n_qpos, gqa, d_model, clips, lam):
    from oracle import optr
    kvq = gu.kvq_lib()
    clips, lam = (F32(clips[0]), F32(clips[1])), F32(lam)
    c = W.optr_head(31, n_tok, n_qpos, gqa, d_model)
    q, k, v, mu = _setup(c)
    gen = np.random.default_rng(5)
    a = gen.normal(0, 0.02, (D, D))
    f64 = lambda x: np.asarray(x, np.float64)
    # keys (Eq. 14)
    lk_o, gk_o = optr.key_loss(a, c.r_k0, f64(q), f64(k), f64(v), f64(c.w_o), f64(mu), clips[0], lam)
    lk_g, gk_g = _gpu_loss_grad(kvq, kvq.KVQ_OPTR_KEYS, q, k, v, c.w_o, mu, c.r_k0, a, None, clips[0], clips[1], lam)
    assert abs(lk_g - lk_o) <= 1e-9 * abs(lk_o), (lk_g, lk_o)
    assert gu.normwise_err(gk_g, gk_o) <= 1e-8, gu.normwise_err(gk_g, gk_o)
    # values (Eq. 16) under the weights of a selected key rotation
    r_sel = optr.rotation(c.r_k0, a)
    p_hat = optr.selected_key_weights(r_sel, f64(q), f64(k), f64(mu), clips[0])
    b = gen.normal(0, 0.02, (D, D))
    lv_o, gv_o = optr.value_loss(b, c.r_v0, p_hat, f64(v), f64(c.w_o), clips[1])
    lv_g, gv_g = _gpu_loss_grad(kvq, kvq.KVQ_OPTR_VALUES, q, k, v, c.w_o, mu, c.r_v0, b, r_sel, clips[0], clips[1],
                                lam)
    assert abs(lv_g - lv_o) <= 1e-9 * abs(lv_o), (lv_g, lv_o)
    assert gu.normwise_err(gv_g, gv_o) <= 1e-8, gu.normwise_err(gv_g, gv_o)
    print(f"keys: loss {lk_g:.6g} (oracle {lk_o:.6g}), grad err {gu.normwise_err(gk_g, gk_o):.2e}; "
          f"values: loss {lv_g:.6g} (oracle {lv_o:.6g}), grad err {gu.normwise_err(gv_g, gv_o):.2e}")


def _gpu_calibrate(kvq, c, mu, clips, steps, lr, every, heldout=True):
    torch = gu.torch_cuda()
    q, k, v = c.train
    qh, kh, vh = c.heldout
    ws = torch.empty(kvq.kvq_optr_workspace_size(k.shape[0], q.shape[0], q.shape[1],
                                                 kh.shape[0] if heldout else 0, qh.shape[0] if heldout else 0),
                     dtype=torch.uint8, device="cuda")
    r_k = torch.zeros(D, D, dtype=torch.float64, device="cuda")
    r_v = torch.zeros_like(r_k)
    lk = torch.zeros(steps, dtype=torch.float64, device="cuda")
    lv = torch.zeros_like(lk)
    tr = (_dev32(q), _dev32(k), _dev32(v))
    ho = (_dev32(qh), _dev32(kh), _dev32(vh)) if heldout else None
    kvq.kvq_optr_calibrate_head(tr, ho, _dev32(c.w_o), _dev32(mu), _dev64(c.r_k0), _dev64(c.r_v0), clips[0], clips[1],
                                1.0, steps, lr, every, r_k, r_v, lk, lv, ws)
    torch.cuda.synchronize()
    kvq.kvq_device_check()
    return r_k.cpu().numpy(), r_v.cpu().numpy(), lk.cpu().numpy(), lv.cpu().numpy()


def test_calibration_run_matches_the_oracle():
    """Algorithm 1 at the paper's rate (0.02), 40 steps per phase, selection every 20
    steps on a held-out trace: the same training losses, the same selected rotations."""
    from oracle import optr
    kvq = gu.kvq_lib()
    c = W.optr_head(32, 48, 6, 2, 16)
    q, k, v, mu = _setup(c)
    clips = (F32(0.96), F32(0.92))
    f64 = lambda x: np.asarray(x, np.float64)
    ho = tuple(f64(x) for x in c.heldout)
    r_k_o, r_v_o, lk_o, lv_o = optr.calibrate_head(f64(q), f64(k), f64(v), f64(c.w_o), c.r_k0, c.r_v0, f64(mu),
                                                   clips[0], clips[1], steps=40, lr=F32(0.02), heldout=ho, every=20)
    r_k, r_v, lk, lv = _gpu_calibrate(kvq, c, mu, clips, 40, 0.02, 20)
    assert np.abs(lk - lk_o).max() <= 1e-7 * np.abs(lk_o).max(), np.abs(lk - lk_o).max()
    assert np.abs(lv - lv_o).max() <= 1e-7 * np.abs(lv_o).max(), np.abs(lv - lv_o).max()
    assert np.abs(r_k - r_k_o).max() <= 1e-8 and np.abs(r_v - r_v_o).max() <= 1e-8
    # R = R0 exp(S) with exp(S) orthogonal: R R^T = R0 R0^T (R0 itself is a float32 rotation)
    assert np.abs(r_k @ r_k.T - c.r_k0 @ c.r_k0.T).max() < 1e-12
    assert np.abs(r_v @ r_v.T - c.r_v0 @ c.r_v0.T).max() < 1e-12


def test_serve14b_shaped_head():
    """A head of the 14B-class serving layer's calibration trace (2,560 tokens, the
    last 64 query positions, 4 query heads, d_model 5,120): objectives and gradients
    against the oracle, then a short run (20 steps per phase, selection every 10 on a
    held-out trace) that must select the same rotations."""
    from oracle import optr
    kvq = gu.kvq_lib()
    c = W.optr_head(33, 2560, 64, 4, 5120)
    q, k, v, mu = _setup(c)
    clips = (F32(0.96), F32(0.92))
    f64 = lambda x: np.asarray(x, np.float64)
    a = np.random.default_rng(6).normal(0, 0.01, (D, D))
    lk_o, gk_o = optr.key_loss(a, c.r_k0, f64(q), f64(k), f64(v), f64(c.w_o), f64(mu), clips[0], 1.0)
    lk_g, gk_g = _gpu_loss_grad(kvq, kvq.KVQ_OPTR_KEYS, q, k, v, c.w_o, mu, c.r_k0, a, None, clips[0], clips[1], 1.0)
    assert abs(lk_g - lk_o) <= 1e-9 * abs(lk_o) and gu.normwise_err(gk_g, gk_o) <= 1e-8
    ho = tuple(f64(x) for x in c.heldout)
    r_k_o, r_v_o, lk_o2, lv_o2 = optr.calibrate_head(f64(q), f64(k), f64(v), f64(c.w_o), c.r_k0, c.r_v0, f64(mu),
                                                     clips[0], clips[1], steps=20, lr=F32(0.02), heldout=ho, every=10)
    r_k, r_v, lk, lv = _gpu_calibrate(kvq, c, mu, clips, 20, 0.02, 10)
    assert np.abs(lk - lk_o2).max() <= 1e-7 * np.abs(lk_o2).max()
    assert np.abs(lv - lv_o2).max() <= 1e-7 * np.abs(lv_o2).max()
    assert np.abs(r_k - r_k_o).max() <= 1e-8 and np.abs(r_v - r_v_o).max() <= 1e-8
