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


# ---------------------------------------------------------------------------
# Closed-form values of the two losses ("Output-Aware Rotation for INT2 KV-Cache
# Quantization", §4.3 Eqs. 12-14 and §4.4 Eqs. 15-16), on heads small enough to
# work by hand.  Two cached tokens, one query at position 1, the query along
# channel 0 and the second key along channel 0 scaled so the exact logits are
# (0, beta); a quantizer stand-in that stores every key as zero makes p^K uniform.
# ---------------------------------------------------------------------------
def _zero_keys(z, clip):
    return np.zeros_like(z), np.ones_like(z)


def _two_token_head(beta, gamma, g=1, d_model=4):
    q = np.zeros((1, g, D))
    q[0, :, 0] = 1.0
    k = np.zeros((2, D))
    k[1, 0] = beta * np.sqrt(D)
    v = np.zeros((2, D))
    v[0, 0] = gamma
    w = np.zeros((d_model, g * D))
    for j in range(g):  # every query head reads the first d_model channels
        w[:, j * D:j * D + d_model] = np.eye(d_model)
    return q, k, v, w


def _p_exact(beta):
    p1 = 1.0 / (1.0 + np.exp(-beta))
    return np.array([1.0 - p1, p1])


@pytest.mark.parametrize("beta", [1.0, -2.5, 4.0])
def test_key_loss_kl_term_closed_form(beta):
    """Values kept equal (v = 0), so e_K = 0 and L_K = D_KL(p || uniform) = log 2 - H(p),
    H the binary entropy of the exact distribution (the direction of Eq. 14: the exact
    distribution p first).  scipy.stats.entropy(p, q) evaluates the same divergence."""
    from scipy.stats import entropy
    q, k, v, w = _two_token_head(beta, 0.0)
    loss, _ = optr.key_loss(np.zeros((D, D)), np.eye(D), q, k, v, w, None, 1.0, lam=1.0, grad=False,
                            qfun=_zero_keys)
    p = _p_exact(beta)
    h = -(p[0] * np.log(p[0]) + p[1] * np.log(p[1]))
    assert abs(loss - (np.log(2.0) - h)) < 1e-14
    assert abs(loss - entropy(p, [0.5, 0.5])) < 1e-14


@pytest.mark.parametrize("lam,d_model", [(1.0, 4), (0.7, 4), (2.0, 16)])
def test_key_loss_output_term_closed_form(lam, d_model):
    """v_0 - v_1 = gamma e_0 and W_O,j = [I | 0]: e_K = (1/2 - p_0) gamma e_0, so
    L_K = D_KL(p || uniform) + lambda_K (1/2 - p_0)^2 gamma^2 / d_model (Eq. 14's
    normalisation by the model width, not by the head dimension)."""
    from scipy.stats import entropy
    beta, gamma = 1.5, 3.0
    q, k, v, w = _two_token_head(beta, gamma, d_model=d_model)
    loss, _ = optr.key_loss(np.zeros((D, D)), np.eye(D), q, k, v, w, None, 1.0, lam=lam, grad=False,
                            qfun=_zero_keys)
    p = _p_exact(beta)
    expect = entropy(p, [0.5, 0.5]) + lam * (0.5 - p[0]) ** 2 * gamma ** 2 / d_model
    assert abs(loss - expect) < 1e-13 * max(1.0, expect)


def test_key_loss_is_a_mean_over_query_heads_and_positions():
    """Eq. 14's expectation over (t, j): two query heads that see the same query and
    the same W_O columns give the one-head loss, not twice it."""
    beta, gamma = 0.8, 2.0
    args = dict(lam=1.0, grad=False, qfun=_zero_keys)
    q1, k, v, w1 = _two_token_head(beta, gamma, g=1)
    q2, _, _, w2 = _two_token_head(beta, gamma, g=2)
    l1, _ = optr.key_loss(np.zeros((D, D)), np.eye(D), q1, k, v, w1, None, 1.0, **args)
    l2, _ = optr.key_loss(np.zeros((D, D)), np.eye(D), q2, k, v, w2, None, 1.0, **args)
    assert abs(l1 - l2) < 1e-15


def test_key_loss_kl_matches_torch_kl_div():
    """With the output term off (lambda_K = 0) and the identity rotation, L_K is the mean
    over (t, j) of KL(p || p^K); torch.nn.functional.kl_div(log p^K, p) evaluates
    exactly that divergence (its target is the first argument of KL)."""
    torch = pytest.importorskip("torch")
    from scipy.special import softmax as sp_softmax
    gen = np.random.default_rng(11)
    n_tok, n_qpos, g = 9, 3, 2
    q = gen.standard_normal((n_qpos, g, D))
    k = gen.standard_normal((n_tok, D)) * 2.0
    v = gen.standard_normal((n_tok, D))
    w = gen.standard_normal((6, g * D))
    mu = k.mean(axis=0)
    loss, _ = optr.key_loss(np.zeros((D, D)), np.eye(D), q, k, v, w, mu, 1.0, lam=0.0, grad=False, qfun=_smooth)
    k_eff = _smooth(k - mu, 1.0)[0]
    kls = []
    for i in range(n_qpos):
        t = n_tok - n_qpos + i
        for j in range(g):
            p = sp_softmax(k[: t + 1] @ q[i, j] / np.sqrt(D))
            pk = sp_softmax(k_eff[: t + 1] @ q[i, j] / np.sqrt(D))
            kls.append(float(torch.nn.functional.kl_div(torch.tensor(np.log(pk)), torch.tensor(p),
                                                        reduction="sum")))
    assert abs(loss - np.mean(kls)) < 1e-13


@pytest.mark.parametrize("c,d_model", [(0.5, 4), (1.25, 8)])
def test_value_loss_closed_form(c, d_model):
    """A quantizer stand-in that shifts channel 0 of every value by c gives v~ - v = c e_0
    for every token, so e_V = c e_0 W_O,j^T = c e_0 whatever the weights p^K (they sum to
    one), and L_V = c^2 / d_model (Eq. 16)."""
    def shift0(z, clip):
        out = z.copy()
        out[:, 0] += c
        return out, np.ones_like(z)
    gen = np.random.default_rng(12)
    n_tok, g = 7, 2
    v = gen.standard_normal((n_tok, D))
    w = np.zeros((d_model, g * D))
    for j in range(g):
        w[:, j * D:j * D + d_model] = np.eye(d_model)
    p_hat = []
    for t in (4, 5, 6):
        for j in range(g):
            x = gen.random(t + 1)
            p_hat.append((j, x / x.sum()))
    loss, _ = optr.value_loss(np.zeros((D, D)), np.eye(D), p_hat, v, w, 1.0, grad=False, qfun=shift0)
    assert abs(loss - c * c / d_model) < 1e-14
