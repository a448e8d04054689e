"""Per-head output-error report (fp64).

Test infrastructure only (see the package header).

"Output-Aware Rotation for INT2 KV-Cache Quantization", Figure 5 (per KV head,
the post-W_O attention-output RMS error as a percentage of plain per-group INT2
without rotation) and the appendix paragraph "Output-space error" (for KV head
h and query head j in G_h, over the last query positions:
Delta y_{t,j} = [p~_{t,j}^T V~ - p_{t,j}^T V] W_O,j^T, averaged as ||.||^2 over
positions and query heads), with the exact split of Eq. 8 into a key-induced
term (p~ - p)^T V W^T and a value-induced term p~^T (V~ - V) W^T.

Readings (the pages leave these open):
* p uses the raw keys; p~ the effective keys of the candidate: centred by mu
  (attention-equivalent, Eq. 24), rotated by R_K, INT2 with clip c_K (Eq. 21),
  met by q R_K (Eq. 26); V~ = Q_2(V R_V; c_V) R_V^T (Eqs. 27-28);
* "plain per-group INT2 without rotation" = identity rotations, no centring,
  the same clip ratios;
* query positions are the last n_qpos of the trace, causal (s <= t), as in the
  calibration sweep;
* per KV head h the report sums over positions and the query heads of G_h:
  E_h = sum ||Delta y||^2, E^K_h, E^V_h (the two Eq. 8 terms), E^naive_h, and
  the reference energy Y_h = sum ||y||^2; RMS % of naive = 100 sqrt(E_h / E^naive_h).

Pinned by tests/test_oracle_report.py.
"""
from __future__ import annotations

import numpy as np

from .attention import softmax
from .output import error_decomposition
from .quant import quant_dequant

D = 128


def _effective(k, v, r_k, r_v, mu, clip_k, clip_v):
    """Effective keys in the rotated basis (with the rotation they meet) and values in the unrotated basis."""
    kc = k - (np.asarray(mu, np.float64)[None] if mu is not None else 0.0)
    xk = np.einsum("thc,hcd->thd", kc, r_k)
    xv = np.einsum("thc,hcd->thd", v, r_v)
    k_rot = quant_dequant(xk, clip_k)
    v_eff = np.einsum("thd,hcd->thc", quant_dequant(xv, clip_v), r_v)  # Q(v R) R^T
    return k_rot, v_eff


def head_error_report(q, k, v, w_o, r_k, r_v, mu, clip_k: float, clip_v: float, gqa: int) -> dict:
    """q [n_qpos, H_q, 128] (queries of the last n_qpos positions), k, v [n_tok, H_kv, 128],
    w_o [d_model, H_q * 128]; r_k, r_v [H_kv, 128, 128].  Returns per-KV-head arrays."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    w = np.asarray(w_o, np.float64)
    n_qpos, hq, _ = q.shape
    n_tok, hkv, _ = k.shape
    eye = np.broadcast_to(np.eye(D), (hkv, D, D))
    cand = _effective(k, v, r_k, r_v, mu, clip_k, clip_v)
    naive = _effective(k, v, eye, eye, None, clip_k, clip_v)
    out = {name: np.zeros(hkv) for name in ("e", "e_key", "e_val", "e_naive", "y")}
    for i in range(n_qpos):
        t = n_tok - n_qpos + i
        for j in range(hq):
            h = j // gqa
            w_j = w[:, j * D:(j + 1) * D]
            p = softmax(k[: t + 1, h] @ q[i, j] / np.sqrt(D))
            out["y"][h] += float((((p @ v[: t + 1, h]) @ w_j.T) ** 2).sum())
            for name, (k_rot, v_eff), r in (("c", cand, r_k), ("n", naive, eye)):
                p_t = softmax(k_rot[: t + 1, h] @ (q[i, j] @ r[h]) / np.sqrt(D))
                dy, dk, dv = error_decomposition(p, p_t, v[: t + 1, h], v_eff[: t + 1, h], w_j)
                if name == "c":
                    out["e"][h] += float((dy ** 2).sum())
                    out["e_key"][h] += float((dk ** 2).sum())
                    out["e_val"][h] += float((dv ** 2).sum())
                else:
                    out["e_naive"][h] += float((dy ** 2).sum())
    out["rms_pct_of_naive"] = 100.0 * np.sqrt(out["e"] / out["e_naive"])
    return out
