"""Pins for oracle.calib: the candidate x clip sweep and its selection rule."""
import numpy as np

from oracle import calib, quant, rotations, output, attention


def _brute_sweep_entry(q, k, v, w, r, clip, mu, gqa, joint):
    """Step by step: centre, rotate, quantize/dequantize, unrotate, attend, project."""
    kt = quant.rotated_quant_dequant(k.reshape(-1, 128) - np.tile(mu, (k.shape[0], 1)) if mu is not None
                                     else k.reshape(-1, 128), r, clip).reshape(k.shape)
    if mu is not None:
        kt = kt + mu[None]
    vt = quant.rotated_quant_dequant(v.reshape(-1, 128), r, clip).reshape(v.shape)
    o = attention.causal_attention(q, kt, vt, gqa)
    o_ref = attention.causal_attention(q, k, v, gqa)
    y = output.out_proj_per_kv_head(o, w, gqa)
    y_ref = output.out_proj_per_kv_head(o_ref, w, gqa)
    if joint:
        y, y_ref = y.sum(axis=-2), y_ref.sum(axis=-2)
        return ((y - y_ref) ** 2).sum() / (y_ref ** 2).sum()
    return ((y - y_ref) ** 2).sum(axis=(0, 2)) / (y_ref ** 2).sum(axis=(0, 2))


def test_sweep_matches_step_by_step_composition():
    g = np.random.default_rng(0)
    n, nq, hkv, gqa, dm = 40, 3, 2, 2, 24
    k = g.standard_normal((n, hkv, 128)) + 6 * (g.random(128) < 0.05)
    v = g.standard_normal((n, hkv, 128))
    q = g.standard_normal((nq, hkv * gqa, 128))
    w = g.standard_normal((dm, hkv * gqa * 128)) / 20
    mu = k.mean(axis=0)
    r1 = rotations.signed_hadamard(np.where(g.random(128) < .5, -1., 1.))
    r2 = rotations.expm_skew(g.normal(0, 0.05, (128, 128)))
    mats = [np.stack([np.eye(128)] * hkv), np.stack([r1] * hkv), np.stack([r2] * hkv)]
    clips = (1.0, 0.85)
    for joint in (False, True):
        nm, err, ref = calib.calib_sweep(q, k, v, w, mats, clips, mu, gqa, joint)
        assert nm.shape == (3, 2, 1 if joint else hkv)
        for i, m in enumerate(mats):
            for c_i, c in enumerate(clips):
                # the brute force rotates every head by the same matrix here
                b = _brute_sweep_entry(q, k, v, w, m[0], c, mu, gqa, joint)
                assert np.abs(nm[i, c_i] - b).max() < 1e-9 * max(1.0, np.abs(b).max())


def test_centring_does_not_change_unquantized_scores_but_helps_int2():
    g = np.random.default_rng(1)
    n, hkv = 64, 1
    k = g.standard_normal((n, hkv, 128))
    k[:, :, :6] += 10.0
    v = g.standard_normal((n, hkv, 128))
    q = g.standard_normal((2, 1, 128))
    w = g.standard_normal((16, 128)) / 10
    mats = [np.eye(128)[None]]
    nm_c, _, _ = calib.calib_sweep(q, k, v, w, mats, (1.0,), k.mean(axis=0), 1, False)
    nm_n, _, _ = calib.calib_sweep(q, k, v, w, mats, (1.0,), None, 1, False)
    assert nm_c[0, 0, 0] < nm_n[0, 0, 0]


def test_select_tie_break():
    nm = np.array([[[2.0], [1.0]], [[1.0], [3.0]]])  # (0,1) and (1,0) tie at 1.0
    assert calib.select(nm) == [(0, 1)]
    nm2 = np.array([[[5.0, 1.0]], [[4.0, 2.0]]])
    assert calib.select(nm2) == [(1, 0), (0, 0)]
