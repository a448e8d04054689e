"""Pins for oracle.optr (Algorithm 1 of the OptR paper on one KV head)."""
import numpy as np
import pytest

from oracle import optr, rotations

D = 128


def _smooth(z, clip):
    """A smooth, non-rotation-invariant stand-in for Q_2 with its exact derivative."""
    return z + 0.2 * np.sin(2.0 * z), 1.0 + 0.4 * np.cos(2.0 * z)


def _head(seed, n_tok=10, n_qpos=3, g=2, dm=12):
    gen = np.random.default_rng(seed)
    q = gen.standard_normal((n_qpos, g, D))
    k = gen.standard_normal((n_tok, D)) * 1.5
    k[:, :3] += 6.0
    v = gen.standard_normal((n_tok, D))
    w = gen.standard_normal((dm, g * D)) / np.sqrt(g * D)
    r0 = rotations.expm_skew(gen.normal(0, 0.1, (D, D)))
    mu = k.mean(axis=0)
    a = gen.normal(0, 0.01, (D, D))
    return gen, q, k, v, w, r0, mu, a


def _directional(fun, a, direction, h=1e-5):
    return (fun(a + h * direction) - fun(a - h * direction)) / (2 * h)


def test_key_gradient_matches_finite_differences():
    gen, q, k, v, w, r0, mu, a = _head(1)
    loss, grad = optr.key_loss(a, r0, q, k, v, w, mu, 1.0, lam=0.7, qfun=_smooth)
    assert loss > 0
    for _ in range(3):
        dirn = gen.standard_normal((D, D))
        fd = _directional(lambda x: optr.key_loss(x, r0, q, k, v, w, mu, 1.0, lam=0.7, grad=False, qfun=_smooth)[0],
                          a, dirn)
        assert abs(fd - np.sum(grad * dirn)) < 1e-6 * (abs(fd) + 1e-12), (fd, np.sum(grad * dirn))


def test_value_gradient_matches_finite_differences():
    gen, q, k, v, w, r0, mu, a = _head(2)
    p_hat = optr.selected_key_weights(r0, q, k, mu, 0.9)
    loss, grad = optr.value_loss(a, r0, p_hat, v, w, 1.0, qfun=_smooth)
    assert loss > 0
    for _ in range(3):
        dirn = gen.standard_normal((D, D))
        fd = _directional(lambda x: optr.value_loss(x, r0, p_hat, v, w, 1.0, grad=False, qfun=_smooth)[0], a, dirn)
        assert abs(fd - np.sum(grad * dirn)) < 1e-6 * (abs(fd) + 1e-12)


def test_straight_through_mask_is_the_clip_range():
    z = np.concatenate([np.linspace(-2, 3, 128)[None], np.linspace(-1, 1, 128)[None]])
    _, m1 = optr.quant_ste(z, 1.0)
    assert np.all(m1 == 1.0)
    _, m = optr.quant_ste(z, 0.8)
    lo, hi = 0.8 * z.min(-1, keepdims=True), 0.8 * z.max(-1, keepdims=True)
    assert np.array_equal(m, ((z >= lo) & (z <= hi)).astype(float))
    assert 0 < m.sum() < m.size


def test_losses_vanish_on_lossless_inputs():
    gen = np.random.default_rng(3)
    n_tok, n_qpos, g = 12, 3, 2
    lo = gen.integers(-16, 0, (n_tok, 1)) / 8.0
    s = gen.integers(1, 8, (n_tok, 1)) / 8.0
    i = gen.integers(0, 4, (n_tok, D))
    i[:, 0], i[:, 1] = 0, 3
    grid = lo + s * i  # rows on a 4-level grid: Q_2 with clip 1 is exact
    q = gen.standard_normal((n_qpos, g, D))
    w = gen.standard_normal((8, g * D))
    eye = np.eye(D)
    lk, _ = optr.key_loss(np.zeros((D, D)), eye, q, grid, grid, w, None, 1.0, grad=False)
    assert abs(lk) < 1e-14
    p_hat = optr.selected_key_weights(eye, q, grid, None, 1.0)
    lv, _ = optr.value_loss(np.zeros((D, D)), eye, p_hat, grid, w, 1.0, grad=False)
    assert abs(lv) < 1e-24


def _trace(gen, n_tok=48, n_qpos=6, g=2):
    q = gen.standard_normal((n_qpos, g, D))
    k = gen.standard_normal((n_tok, D))
    k[:, :6] += np.array([10.0, -10.0, 10.0, 10.0, -10.0, 10.0])
    v = gen.standard_normal((n_tok, D))
    v[:, :2] *= 6.0
    return q, k, v


def test_straight_through_gradient_descends_at_a_small_rate():
    """Algorithm 1's updates lower both training losses at a small learning rate."""
    gen = np.random.default_rng(4)
    n_tok, n_qpos, g, dm = 48, 6, 2, 16
    q = gen.standard_normal((n_qpos, g, D))
    k = gen.standard_normal((n_tok, D))
    k[:, :6] += gen.choice([-10.0, 10.0], 6)
    v = gen.standard_normal((n_tok, D))
    v[:, :2] *= 6.0
    w = gen.standard_normal((dm, g * D)) / np.sqrt(g * D)
    r0 = rotations.expm_skew(gen.normal(0, 0.05, (D, D)))
    mu = k.mean(axis=0)
    _, _, lk, lv = optr.calibrate_head(q, k, v, w, r0, r0, mu, 0.96, 0.92, steps=12, lr=0.001, every=1000)
    assert lk[-1] < 0.7 * lk[0] and lv[-1] < 0.7 * lv[0]


def test_selection_never_returns_worse_than_the_base_rotation_on_held_out_data():
    """At the paper's rate (0.02) the iterates oscillate; the selection every 20 steps
    (step 0 included) keeps the held-out loss at or below the base rotation's, and the
    selected rotations stay orthogonal."""
    gen = np.random.default_rng(5)
    q, k, v = _trace(gen)
    qh, kh, vh = _trace(gen)
    w = gen.standard_normal((16, 2 * D)) / np.sqrt(2 * D)
    r0 = rotations.expm_skew(gen.normal(0, 0.05, (D, D)))
    mu = k.mean(axis=0)
    r_k, r_v, lk, lv = optr.calibrate_head(q, k, v, w, r0, r0, mu, 0.96, 0.92, steps=40, heldout=(qh, kh, vh))
    assert len(lk) == len(lv) == 40
    for r in (r_k, r_v):
        assert np.abs(r @ r.T - np.eye(D)).max() < 1e-12
    zero = np.zeros((D, D))
    base_k = optr.key_loss(zero, r0, qh, kh, vh, w, mu, 0.96, grad=False)[0]
    sel_k = optr.key_loss(np.zeros((D, D)), r_k, qh, kh, vh, w, mu, 0.96, grad=False)[0]
    assert sel_k <= base_k * (1 + 1e-12)
    p_sel = optr.selected_key_weights(r_k, qh, kh, mu, 0.96)
    base_v = optr.value_loss(zero, r0, p_sel, vh, w, 0.92, grad=False)[0]
    sel_v = optr.value_loss(zero, r_v, p_sel, vh, w, 0.92, grad=False)[0]
    assert sel_v <= base_v * (1 + 1e-12)
