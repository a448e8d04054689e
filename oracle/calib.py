"""Candidate-rotation x clip-ratio sweep scored by post-W_O NMSE (fp64).

Test infrastructure only (see the package header).

"Output-aware INT2 KV-cache rotation evaluation": the identity baseline and each
signed-Hadamard candidate search clip ratios on calibration queries; candidate
selection minimises calibration post-W_O NMSE.  "Output-Aware Rotation for INT2
KV-Cache Quantization" (Appendix, Calibration details): the objective is taken
over the final 64 query positions; rotations are selected per KV head.

Readings (the pages leave them open):
* a candidate R is applied to the keys and the values of every KV head, and one
  clip ratio c to both (the evaluation page names one rotation and one clip per
  row);
* keys are centred by mu before the rotation (§4.1) when mu is given;
* query positions are the last n_qpos of the n_tok-token trace, causal (s <= t);
* per-head mode scores y_h = sum_{j in G_h} o_j W_O,j^T; joint mode scores the
  sum over heads; the pooled NMSE is sum_t ||y~_t - y_t||^2 / sum_t ||y_t||^2;
* argmin ties go to the lowest candidate index, then the earlier clip.

Pinned by tests/test_oracle_calib.py (composition against the step-by-step
oracle functions, and against brute force on a tiny case).
"""
from __future__ import annotations

import numpy as np

from .attention import causal_attention, rotate_queries
from .cache import rotate_heads
from .output import out_proj_per_kv_head
from .quant import quant_dequant

D = 128


def calib_sweep(q, k, v, w_o, cand_mats, clips, mu, gqa: int, joint: bool):
    """Returns (nmse [n_cand, n_clip, H], err [n_cand, n_clip, H], ref [H]) with H = 1 if joint."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    w = np.asarray(w_o, np.float64)
    hkv = k.shape[1]
    o_ref = causal_attention(q, k, v, gqa)
    y_ref = out_proj_per_kv_head(o_ref, w, gqa)  # [n_qpos, Hkv, d_model]
    if joint:
        y_ref = y_ref.sum(axis=-2, keepdims=True)
    ref = (y_ref ** 2).sum(axis=(0, 2))
    kc = k - (np.asarray(mu, np.float64)[None] if mu is not None else 0.0)
    n_c = len(cand_mats)
    err = np.zeros((n_c, len(clips), y_ref.shape[1]))
    for i, r in enumerate(cand_mats):
        xk = rotate_heads(kc, r)
        xv = rotate_heads(v, r)
        qr = rotate_queries(q, r, gqa)
        for c_i, c in enumerate(clips):
            kh = quant_dequant(xk, c)
            vh = quant_dequant(xv, c)
            o_rot = causal_attention(qr, kh, vh, gqa)
            # back to the unrotated value basis (equivalently, use W_O R as Eq. 29 folds it)
            o = np.einsum("tjd,jcd->tjc", o_rot, r[np.arange(q.shape[1]) // gqa])
            y = out_proj_per_kv_head(o, w, gqa)
            if joint:
                y = y.sum(axis=-2, keepdims=True)
            err[i, c_i] = ((y - y_ref) ** 2).sum(axis=(0, 2))
    return err / ref[None, None, :], err, ref


def select(nmse: np.ndarray) -> list[tuple[int, int]]:
    """Argmin (candidate, clip) per head column; ties -> lowest candidate, then clip."""
    out = []
    n_c, n_k, n_h = nmse.shape
    for h in range(n_h):
        best = None
        for i in range(n_c):
            for c in range(n_k):
                if best is None or nmse[i, c, h] < nmse[best[0], best[1], h]:
                    best = (i, c)
        out.append(best)
    return out
