"""Post-W_O output, W_O folding, NMSE and the exact error decomposition (fp64).

Test infrastructure only (see the package header).

"Output-Aware Rotation for INT2 KV-Cache Quantization":
* Eq. 3: y_j = o_j W_O,j^T with W_O,j in R^{d_model x d} the columns
  [j*d, (j+1)*d) of W_O in R^{d_model x H_q d}; the layer output sums over j.
* Eqs. 29-31: W_O,j-bar = W_O,j R_V,h(j), and (o_j R_V) W_O,j-bar^T = o_j W_O,j^T.
* Eq. 8: y~ - y = (sum_s dp_s v_s) W_O^T + (sum_s p~_s dv_s) W_O^T exactly.
* Eq. 10 / the evaluation page: post-W_O NMSE = ||y~ - y||^2 / ||y||^2 (a plain
  ratio: the page reports values above 1); summary = mean and *population*
  standard deviation over queries; threshold quality = mean of 1{NMSE <= 10}.

Pinned by tests/test_oracle_output.py.
"""
from __future__ import annotations

import numpy as np

D = 128


def fold_wo(w_o: np.ndarray, r_v: np.ndarray, gqa: int) -> np.ndarray:
    """W_O-bar [d_model, H_q*128] with block j = W_O,j @ R_V,h(j)."""
    w = np.asarray(w_o, np.float64)
    hq = w.shape[1] // D
    out = np.empty_like(w)
    for j in range(hq):
        out[:, j * D:(j + 1) * D] = w[:, j * D:(j + 1) * D] @ r_v[j // gqa]
    return out


def out_proj(o: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = sum_j o_j W_j^T for o [..., H_q, 128], w [d_model, H_q*128] -> [..., d_model]."""
    o = np.asarray(o, np.float64)
    w = np.asarray(w, np.float64)
    hq = o.shape[-2]
    y = 0.0
    for j in range(hq):
        y = y + o[..., j, :] @ w[:, j * D:(j + 1) * D].T
    return y


def out_proj_per_kv_head(o: np.ndarray, w: np.ndarray, gqa: int) -> np.ndarray:
    """y_h = sum_{j in G_h} o_j W_j^T -> [..., H_kv, d_model]."""
    o = np.asarray(o, np.float64)
    hq = o.shape[-2]
    hkv = hq // gqa
    return np.stack([out_proj(o[..., h * gqa:(h + 1) * gqa, :], np.asarray(w, np.float64)[:, h * gqa * D:(h + 1) * gqa * D])
                     for h in range(hkv)], axis=-2)


def nmse(y: np.ndarray, y_ref: np.ndarray) -> float:
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    return float(((y - y_ref) ** 2).sum() / (y_ref ** 2).sum())


def mean_popsd(values) -> tuple[float, float]:
    x = np.asarray(values, np.float64)
    m = x.mean()
    return float(m), float(np.sqrt(((x - m) ** 2).mean()))


def threshold_rate(nmses, threshold: float = 10.0) -> tuple[float, float]:
    return mean_popsd((np.asarray(nmses) <= threshold).astype(np.float64))


def error_decomposition(p, p_tilde, v, v_tilde, w_j):
    """Eq. 8 for one query head: returns (dy, key-induced term, value-induced term)."""
    p = np.asarray(p, np.float64)
    p_tilde = np.asarray(p_tilde, np.float64)
    v = np.asarray(v, np.float64)
    v_tilde = np.asarray(v_tilde, np.float64)
    w_j = np.asarray(w_j, np.float64)
    y = (p @ v) @ w_j.T
    y_tilde = (p_tilde @ v_tilde) @ w_j.T
    dk = ((p_tilde - p) @ v) @ w_j.T
    dv = (p_tilde @ (v_tilde - v)) @ w_j.T
    return y_tilde - y, dk, dv
