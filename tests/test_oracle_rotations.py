"""Pins for oracle.rotations (Hadamard, signed Hadamard, skew exponential)."""
import numpy as np
import pytest
import scipy.linalg

from oracle import rotations


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
def test_sylvester_matches_scipy_and_is_orthogonal(n):
    h = rotations.sylvester_hadamard(n)
    assert np.array_equal(h, scipy.linalg.hadamard(n))
    assert np.array_equal(h @ h.T, n * np.eye(n))


def _fwht(x):
    """Independent in-place fast Walsh-Hadamard transform (butterflies), unnormalised."""
    x = np.array(x, dtype=np.float64)
    n = x.shape[-1]
    h = 1
    while h < n:
        for i in range(0, n, 2 * h):
            a = x[..., i:i + h].copy()
            b = x[..., i + h:i + 2 * h].copy()
            x[..., i:i + h] = a + b
            x[..., i + h:i + 2 * h] = a - b
        h *= 2
    return x


def test_signed_hadamard_orthogonal_and_equals_fwht_of_signed_input():
    g = np.random.default_rng(0)
    s = np.where(g.random(128) < 0.5, -1.0, 1.0)
    r = rotations.signed_hadamard(s)
    assert np.abs(r @ r.T - np.eye(128)).max() < 1e-12
    x = g.standard_normal((5, 128))
    # x R = FWHT(x * s) / sqrt(128): signs applied to input channels first
    assert np.abs(x @ r - _fwht(x * s) / np.sqrt(128)).max() < 1e-12
    # a sign on the wrong side (output channels) would differ
    assert np.abs(x @ r - (_fwht(x) / np.sqrt(128)) * s).max() > 1e-3


def test_expm_skew_matches_scipy():
    g = np.random.default_rng(1)
    for n, std in ((128, 0.05), (16, 1.0), (4, 3.0)):
        a = g.normal(0, std, (n, n))
        ref = scipy.linalg.expm(a - a.T)
        got = rotations.expm_skew(a)
        assert np.abs(got - ref).max() < 1e-11 * max(1.0, np.abs(ref).max())


def test_expm_skew_closed_form_2x2():
    # A - A^T = [[0, t], [-t, 0]]  ->  exp = [[cos t, sin t], [-sin t, cos t]]
    for t in (0.3, 1.0, 2.5, -4.0):
        a = np.array([[0.0, t], [0.0, 0.0]])
        r = rotations.expm_skew(a)
        ref = np.array([[np.cos(t), np.sin(t)], [-np.sin(t), np.cos(t)]])
        assert np.abs(r - ref).max() < 1e-13


def test_expm_skew_is_special_orthogonal():
    g = np.random.default_rng(2)
    a = g.normal(0, 0.05, (128, 128))
    r = rotations.expm_skew(a)
    assert np.abs(r @ r.T - np.eye(128)).max() < 1e-12
    sign, logdet = np.linalg.slogdet(r)
    assert sign == 1.0 and abs(logdet) < 1e-10


def test_rotation_matrices_dispatch():
    g = np.random.default_rng(3)
    s = np.where(g.random((3, 128)) < 0.5, -1.0, 1.0)
    rs = rotations.rotation_matrices("signed_hadamard", 3, signs=s)
    assert rs.shape == (3, 128, 128)
    assert np.allclose(rs[1], rotations.signed_hadamard(s[1]))
    assert np.array_equal(rotations.rotation_matrices("identity", 2)[1], np.eye(128))
