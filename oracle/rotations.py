"""Orthogonal rotations used by the method (fp64).

Test infrastructure only (see the package header).

* ``sylvester_hadamard(n)``: H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]].  The
  QuaRot-style base rotation named in "Output-Aware Rotation for INT2 KV-Cache
  Quantization" (§2, Baselines of §5) and the "deterministic signed-Hadamard
  candidates" of "Output-aware INT2 KV-cache rotation evaluation".
  Pinned: equals scipy.linalg.hadamard; H H^T = n I.
* ``signed_hadamard(s)``: R = diag(s) H / sqrt(n) (the sign vector multiplies the
  input channels before the transform).  Pinned: R R^T = I.
* ``expm_skew(A)``: R = exp(A - A^T) (§4.2, Eq. 11) by scaling and squaring of a
  Taylor series (Moler & Van Loan, "Nineteen dubious ways to compute the
  exponential of a matrix", methods 1 and 3).  Pinned: scipy.linalg.expm, the
  closed-form 2x2 rotation, R R^T = I and det R = +1.
"""
from __future__ import annotations

import numpy as np

D = 128


def sylvester_hadamard(n: int) -> np.ndarray:
    assert n >= 1 and (n & (n - 1)) == 0, "n must be a power of two"
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def signed_hadamard(signs: np.ndarray) -> np.ndarray:
    """R = diag(signs) @ H / sqrt(n); a row vector x is rotated as x @ R."""
    s = np.asarray(signs, dtype=np.float64)
    n = s.shape[-1]
    return (s[:, None] * sylvester_hadamard(n)) / np.sqrt(n)


def expm_skew(a: np.ndarray, tol: float = 1e-17) -> np.ndarray:
    """exp(A - A^T) by scaling and squaring with a Taylor series."""
    a = np.asarray(a, dtype=np.float64)
    s_mat = a - a.T
    norm = np.abs(s_mat).sum(axis=1).max()  # infinity norm
    k = 0
    while norm / (2 ** k) > 0.5:
        k += 1
    x = s_mat / (2 ** k)
    n = x.shape[0]
    result = np.eye(n)
    term = np.eye(n)
    j = 1
    while True:
        term = term @ x / j
        result = result + term
        if np.abs(term).max() < tol:
            break
        j += 1
    for _ in range(k):
        result = result @ result
    return result


def rotation_matrices(kind: str, n_heads: int, signs=None, dense=None) -> np.ndarray:
    """Per-head rotation matrices [n_heads, 128, 128] in fp64 from a rotation spec."""
    if kind == "identity":
        return np.broadcast_to(np.eye(D), (n_heads, D, D)).copy()
    if kind == "signed_hadamard":
        s = np.asarray(signs, dtype=np.float64)
        assert s.shape == (n_heads, D)
        return np.stack([signed_hadamard(s[h]) for h in range(n_heads)])
    if kind == "dense":
        r = np.asarray(dense, dtype=np.float64)
        assert r.shape == (n_heads, D, D)
        return r.copy()
    raise ValueError(kind)


def rot_matrices(rot, n_heads: int) -> np.ndarray:
    """Same, from a ``workloads.Rot``-like object (attributes kind, signs, dense)."""
    return rotation_matrices(rot.kind, n_heads, getattr(rot, "signs", None), getattr(rot, "dense", None))
