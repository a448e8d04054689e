"""OptR offline calibration of one KV head: losses, straight-through gradients,
Adam (fp64).

Test infrastructure only (see the package header).

"Output-Aware Rotation for INT2 KV-Cache Quantization": §4.2 Eq. 11 (R = R^0
exp(A - A^T)), §4.3 Eqs. 12-14 (key loss: KL(p || p^K) + lambda_K ||e_K||^2 /
d_model, values kept exact), §4.4 Eqs. 15-16 (value loss ||e_V||^2 / d_model
under the selected key path), §4.5 Eqs. 17-18 (INT2 quantization in the loop,
straight-through estimator), Algorithm 1 (keys first for T steps, then values),
§5 implementation details (lambda_K = 1, 80 Adam steps, learning rate 0.02).

Readings (the pages leave these open):
* The straight-through estimator passes the gradient of a quantized channel iff
  it lies inside its group's clip range [c min, c max] (Eq. 18's |Z| <= tau_c
  for the asymmetric quantizer); the scale and zero are treated as constants.
* Expectations over (t, j) are plain means over the query positions (the last
  n_qpos of the trace, causal) and the query heads of the KV head.
* Adam uses the common defaults beta1 = 0.9, beta2 = 0.999, eps = 1e-8.
* Selection "every 20 steps" (§5, appendix calibration details): the iterates
  after 0, 20, 40, ... steps are candidates (step 0 = the base rotation), scored
  by the same loss on a held-out split when one is given, else on the training
  trace; the lowest wins (ties to the earlier step).  Each Adam step moves every
  generator entry by about the learning rate, so at the paper's 0.02 the losses
  of a synthetic head oscillate and the selection matters.
* Gradients of exp(S) use the Frechet derivative (SciPy's expm_frechet):
  dL/dS = Dexp(S^T)[dL/dE], then dL/dA = dL/dS - (dL/dS)^T.

Pinned by tests/test_oracle_optr.py: closed-form values of both losses on
two-token heads worked by hand (KL against uniform = log 2 minus the binary
entropy, with scipy.stats.entropy as a second evaluator; the output term's
lambda_K (1/2 - p_0)^2 gamma^2 / d_model; the value loss c^2 / d_model for a
constant shift; the mean over query heads), the KL term against
torch.nn.functional.kl_div, the analytic gradients against central finite
differences with a smooth stand-in for the quantizer (so the whole chain --
softmax, KL, e_K / e_V, rotations, the exponential's Frechet derivative -- is
differentiable), the straight-through mask, zero losses on lossless inputs,
orthogonality of the iterates, loss decrease under Algorithm 1.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import expm, expm_frechet

from .attention import softmax
from .quant import quantize_groups

D = 128


def rotation(r0: np.ndarray, a: np.ndarray) -> np.ndarray:
    """Eq. 11: R = R^0 exp(A - A^T)."""
    return r0 @ expm(a - a.T)


def quant_ste(z: np.ndarray, clip: float):
    """Dequantized Q_2(z) per row group of 128 and the straight-through derivative of
    Eq. 18 (1 inside the group's clip range, 0 outside).  Any map returning
    (value, elementwise derivative) can stand in for it (the pins use a smooth one)."""
    codes, s, zero = quantize_groups(z, clip)
    zq = zero[..., None] + s[..., None] * codes.astype(np.float64)
    lo = clip * z.min(axis=-1, keepdims=True)
    hi = clip * z.max(axis=-1, keepdims=True)
    mask = ((z >= lo) & (z <= hi)).astype(np.float64)
    return zq, mask


def kl_term(p: np.ndarray, pk: np.ndarray):
    """Eq. 14's D_KL(p_t || p_t^K) = sum_s p_s log(p_s / p^K_s) (the exact attention
    distribution first) and its gradient with respect to the logits a^K of
    p^K = softmax(a^K): p^K - p."""
    return float(np.sum(p * (np.log(p) - np.log(pk)))), pk - p


def output_error_term(e: np.ndarray, d_model: int):
    """The post-W_O error term of Eqs. 14 and 16, ||e||_2^2 / d_model, and its gradient 2 e / d_model."""
    return float(e @ e) / d_model, (2.0 / d_model) * e


def _positions(n_tok: int, n_qpos: int):
    return [n_tok - n_qpos + i for i in range(n_qpos)]


def key_loss(a, r0, q, k, v, w_o, mu, clip: float, lam: float = 1.0, grad: bool = True, qfun=quant_ste):
    """L_K (Eq. 14) of one KV head and dL_K/dA.

    q [n_qpos, G, 128] (queries of the last n_qpos positions), k, v [n_tok, 128],
    w_o [d_model, G * 128] (the W_O columns of the head's query heads)."""
    s_mat = a - a.T
    e_mat = expm(s_mat)
    r = r0 @ e_mat
    n_qpos, g, _ = q.shape
    n_tok = k.shape[0]
    dm = w_o.shape[0]
    x = k - (mu if mu is not None else 0.0)
    z = x @ r
    zq, mask = qfun(z, clip)
    k_eff = zq @ r.T  # effective keys, unrotated basis
    n = n_qpos * g
    loss = 0.0
    g_keff = np.zeros_like(k_eff)  # dL/dk~_s
    for i, t in enumerate(_positions(n_tok, n_qpos)):
        for j in range(g):
            qq = q[i, j]
            w_j = w_o[:, j * D:(j + 1) * D]
            a_ref = k[: t + 1] @ qq / np.sqrt(D)
            a_k = k_eff[: t + 1] @ qq / np.sqrt(D)
            p = softmax(a_ref)
            pk = softmax(a_k)
            kl, dkl = kl_term(p, pk)
            vt = v[: t + 1]
            e = ((pk - p) @ vt) @ w_j.T  # Eq. 13: [sum_s (p^K_s - p_s) v_s] W_j^T
            err, derr = output_error_term(e, dm)
            loss += (kl + lam * err) / n
            if grad:
                dpk = lam * (vt @ (w_j.T @ derr))  # d(lam ||e||^2 / dm) / dp^K_s = lam v_s . W_j^T derr
                da = pk * (dpk - pk @ dpk) + dkl  # softmax backward, plus dKL/da^K
                g_keff[: t + 1] += np.outer(da / n, qq) / np.sqrt(D)
    if not grad:
        return loss, None
    # k~ = zq R^T, zq = Q(z) (straight-through), z = x R
    d_r = g_keff.T @ zq  # via R^T: sum_s G_s zq_s^T
    d_zq = g_keff @ r
    d_r += x.T @ (d_zq * mask)
    d_e = r0.T @ d_r
    d_s = expm_frechet(s_mat.T, d_e, compute_expm=False)
    return loss, d_s - d_s.T


def value_loss(a, r0, p_hat, v, w_o, clip: float, grad: bool = True, qfun=quant_ste):
    """L_V (Eq. 16) of one KV head and dL_V/dA.

    p_hat: list over (position i, query head j) of the selected key path's
    weights p^K_t [t + 1]; v [n_tok, 128]; w_o [d_model, G * 128]."""
    s_mat = a - a.T
    e_mat = expm(s_mat)
    r = r0 @ e_mat
    dm = w_o.shape[0]
    z = v @ r
    zq, mask = qfun(z, clip)
    v_eff = zq @ r.T
    dv = v_eff - v
    n = len(p_hat)
    loss = 0.0
    g_veff = np.zeros_like(v_eff)
    for (j, pk) in p_hat:
        w_j = w_o[:, j * D:(j + 1) * D]
        m = len(pk)
        e = (pk @ dv[:m]) @ w_j.T
        err, derr = output_error_term(e, dm)
        loss += err / n
        if grad:
            g_veff[:m] += np.outer(pk, (derr / n) @ w_j)
    if not grad:
        return loss, None
    d_r = g_veff.T @ zq
    d_zq = g_veff @ r
    d_r += v.T @ (d_zq * mask)
    d_e = r0.T @ d_r
    d_s = expm_frechet(s_mat.T, d_e, compute_expm=False)
    return loss, d_s - d_s.T


def selected_key_weights(r_k, q, k, mu, clip: float):
    """p^K_t of the selected key rotation (Algorithm 1: the key path the value phase uses), tagged with the query head."""
    n_qpos, g, _ = q.shape
    n_tok = k.shape[0]
    x = k - (mu if mu is not None else 0.0)
    zq, _ = quant_ste(x @ r_k, clip)
    k_eff = zq @ r_k.T
    out = []
    for i, t in enumerate(_positions(n_tok, n_qpos)):
        for j in range(g):
            out.append((j, softmax(k_eff[: t + 1] @ q[i, j] / np.sqrt(D))))
    return out


class Adam:
    def __init__(self, shape, lr: float = 0.02, b1: float = 0.9, b2: float = 0.999, eps: float = 1e-8):
        self.m = np.zeros(shape)
        self.v = np.zeros(shape)
        self.t = 0
        self.lr, self.b1, self.b2, self.eps = lr, b1, b2, eps

    def step(self, x, grad):
        self.t += 1
        self.m = self.b1 * self.m + (1 - self.b1) * grad
        self.v = self.b2 * self.v + (1 - self.b2) * grad * grad
        mh = self.m / (1 - self.b1 ** self.t)
        vh = self.v / (1 - self.b2 ** self.t)
        return x - self.lr * mh / (np.sqrt(vh) + self.eps)


def _run_phase(loss_grad, score, steps: int, lr: float, every: int):
    """Adam on A from 0; candidates every `every` steps (and step 0); the best score wins."""
    a = np.zeros((D, D))
    opt = Adam(a.shape, lr)
    losses = []
    best_a, best = a.copy(), score(a)
    for i in range(1, steps + 1):
        loss, gr = loss_grad(a)
        losses.append(loss)
        a = opt.step(a, gr)
        if i % every == 0:
            sc = score(a)
            if sc < best:
                best_a, best = a.copy(), sc
    return best_a, np.array(losses)


def calibrate_head(q, k, v, w_o, r_k0, r_v0, mu, clip_k: float, clip_v: float, steps: int = 80,
                   lr: float = 0.02, lam: float = 1.0, heldout=None, every: int = 20):
    """Algorithm 1 for one KV head: T key steps, then T value steps, each phase
    selecting among its iterates every `every` steps.

    heldout: optional (q, k, v) of a held-out trace for the selection.
    Returns (R_K, R_V, key training losses [steps], value training losses [steps])."""
    qs, ks, vs = heldout if heldout is not None else (q, k, v)
    a_k, lk = _run_phase(lambda a: key_loss(a, r_k0, q, k, v, w_o, mu, clip_k, lam),
                         lambda a: key_loss(a, r_k0, qs, ks, vs, w_o, mu, clip_k, lam, grad=False)[0],
                         steps, lr, every)
    r_k = rotation(r_k0, a_k)
    p_hat = selected_key_weights(r_k, q, k, mu, clip_k)
    p_sel = selected_key_weights(r_k, qs, ks, mu, clip_k)
    a_v, lv = _run_phase(lambda a: value_loss(a, r_v0, p_hat, v, w_o, clip_v),
                         lambda a: value_loss(a, r_v0, p_sel, vs, w_o, clip_v, grad=False)[0],
                         steps, lr, every)
    return r_k, rotation(r_v0, a_v), lk, lv
