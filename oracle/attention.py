"""Decode attention by definition (fp64).

Test infrastructure only (see the package header).

"Output-Aware Rotation for INT2 KV-Cache Quantization", §3 (Eqs. 1-2):
a_s = <q, k_s> / sqrt(d), p = softmax_{s<=t}(a), o = sum_s p_s v_s; with INT2
keys (Eq. 5) the logits use the effective keys.  The cache stores rotated keys
k_R = Q_2((k - mu) R_K) and the query is rotated once instead (appendix
"Rotated-query implementation", Eqs. 21-22 and 26: q k~^T = (q R_K) k_R^T);
values are stored rotated, v' = v R_V, so the attention readout is o' = o R_V
(Eq. 27) and stays in the rotated basis until W_O (Eq. 31).

Query head j reads KV head h(j) = j // g with g = H_q / H_kv (the pages define
only the set G_h of query heads sharing KV head h; this is the standard GQA
grouping).

``split_decode_attention`` evaluates the same softmax over contiguous token
ranges and merges them with the log-sum-exp rule (running max m, sum l,
unnormalised accumulator); it must equal the unsplit result to rounding.

Pinned by tests/test_oracle_attention.py: pure-Python loop brute force on tiny
inputs, Eq. 22/26 equality, Eq. 24 centring invariance, split == unsplit.
"""
from __future__ import annotations

import numpy as np

D = 128


def softmax(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, np.float64)
    m = a.max(axis=-1, keepdims=True)
    e = np.exp(a - m)
    return e / e.sum(axis=-1, keepdims=True)


def rotate_queries(q: np.ndarray, r_k: np.ndarray, gqa: int) -> np.ndarray:
    """q' _j = q_j R_K,h(j) for q [..., H_q, 128]."""
    q = np.asarray(q, np.float64)
    idx = np.arange(q.shape[-2]) // gqa
    return np.einsum("...jc,jcd->...jd", q, r_k[idx])


def decode_attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, r_k: np.ndarray,
                     gqa: int) -> np.ndarray:
    """One query per query head against a whole (dequantized, rotated) cache.

    q [H_q, 128]; k_hat, v_hat [L, H_kv, 128] in the rotated basis;
    returns o' [H_q, 128] in the rotated-V basis.
    """
    qr = rotate_queries(q, r_k, gqa)
    hq = qr.shape[0]
    out = np.empty((hq, D))
    for j in range(hq):
        h = j // gqa
        a = k_hat[:, h, :] @ qr[j] / np.sqrt(D)
        p = softmax(a)
        out[j] = p @ v_hat[:, h, :]
    return out


def split_decode_attention(q, k_hat, v_hat, r_k, gqa: int, n_splits: int) -> np.ndarray:
    """The same readout computed over n_splits contiguous token ranges and merged."""
    qr = rotate_queries(q, r_k, gqa)
    hq = qr.shape[0]
    length = k_hat.shape[0]
    bounds = np.linspace(0, length, n_splits + 1).round().astype(int)
    out = np.empty((hq, D))
    for j in range(hq):
        h = j // gqa
        ms, ls, accs = [], [], []
        for i in range(n_splits):
            lo, hi = bounds[i], bounds[i + 1]
            if hi <= lo:
                continue
            a = k_hat[lo:hi, h, :] @ qr[j] / np.sqrt(D)
            m = a.max()
            e = np.exp(a - m)
            ms.append(m)
            ls.append(e.sum())
            accs.append(e @ v_hat[lo:hi, h, :])
        m_star = max(ms)
        w = [np.exp(m - m_star) for m in ms]
        l_star = sum(wi * li for wi, li in zip(w, ls))
        out[j] = sum(wi * ai for wi, ai in zip(w, accs)) / l_star
    return out


def reference_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, gqa: int) -> np.ndarray:
    """Unquantized, unrotated, uncentred readout o_j (Eqs. 1-2) for q [H_q,128], k, v [L,H_kv,128]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    hq = q.shape[0]
    out = np.empty((hq, D))
    for j in range(hq):
        h = j // gqa
        p = softmax(k[:, h, :] @ q[j] / np.sqrt(D))
        out[j] = p @ v[:, h, :]
    return out


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, gqa: int) -> np.ndarray:
    """Queries at the last n_qpos positions of an n_tok-token trace, causal (s <= t).

    q [n_qpos, H_q, 128] (already in the basis of k), k, v [n_tok, H_kv, 128]
    -> o [n_qpos, H_q, 128].
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n_qpos, hq, _ = q.shape
    n_tok = k.shape[0]
    out = np.empty((n_qpos, hq, D))
    for i in range(n_qpos):
        t = n_tok - n_qpos + i
        for j in range(hq):
            h = j // gqa
            p = softmax(k[: t + 1, h, :] @ q[i, j] / np.sqrt(D))
            out[i, j] = p @ v[: t + 1, h, :]
    return out
