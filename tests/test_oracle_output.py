"""Pins for oracle.output: W_O fold (Eq. 31), projection, NMSE, Eq. 8, statistics."""
import json
import os

import numpy as np

from oracle import output, rotations, attention, quant
from conftest import GOLDEN


def test_folded_wo_reproduces_unrotated_output():
    # Eq. 31: (o_j R_V,h) W_O,j-bar^T = o_j W_O,j^T
    g = np.random.default_rng(0)
    hq, hkv, dm = 4, 2, 96
    w = g.standard_normal((dm, hq * 128))
    rv = np.stack([rotations.expm_skew(g.normal(0, 0.05, (128, 128))) for _ in range(hkv)])
    o = g.standard_normal((3, hq, 128))
    o_rot = np.einsum("bjc,jcd->bjd", o, rv[np.arange(hq) // 2])
    wb = output.fold_wo(w, rv, 2)
    assert np.abs(output.out_proj(o_rot, wb) - output.out_proj(o, w)).max() < 1e-11


def test_out_proj_brute_force():
    g = np.random.default_rng(1)
    hq, dm = 3, 5
    w = g.standard_normal((dm, hq * 128))
    o = g.standard_normal((hq, 128))
    y = [sum(o[j, c] * w[r, j * 128 + c] for j in range(hq) for c in range(128)) for r in range(dm)]
    assert np.abs(output.out_proj(o, w) - np.array(y)).max() < 1e-12
    # per-KV-head outputs sum to the full output
    yh = output.out_proj_per_kv_head(o[None].repeat(2, 0)[:, :2], w[:, :256], 1)
    assert np.abs(yh.sum(axis=-2) - output.out_proj(o[None].repeat(2, 0)[:, :2], w[:, :256])).max() < 1e-12


def test_exact_error_decomposition():
    # Eq. 8: y~ - y = key-induced + value-induced, exactly
    g = np.random.default_rng(2)
    n = 64
    k = g.standard_normal((n, 128)) + 5 * (g.random(128) < 0.05)
    v = g.standard_normal((n, 128))
    q = g.standard_normal(128)
    r = rotations.signed_hadamard(np.where(g.random(128) < .5, -1., 1.))
    kt = quant.rotated_quant_dequant(k, r, 1.0)
    vt = quant.rotated_quant_dequant(v, r, 0.9)
    p = attention.softmax(k @ q / np.sqrt(128))
    pt = attention.softmax(kt @ q / np.sqrt(128))
    w = g.standard_normal((32, 128))
    dy, dk, dv = output.error_decomposition(p, pt, v, vt, w)
    assert np.abs(dy - (dk + dv)).max() < 1e-12
    assert np.abs(dk).max() > 1e-4 and np.abs(dv).max() > 1e-4  # both terms present


def test_nmse_definition():
    y = np.array([3.0, 4.0])
    assert output.nmse(y + np.array([0.0, 1.0]), y) == 1.0 / 25.0
    assert output.nmse(3 * y, y) == 4.0  # a plain ratio, may exceed 1


def test_population_sd_matches_threshold_rows_of_the_evaluation_page():
    with open(os.path.join(GOLDEN, "evaluation_page.json")) as f:
        page = json.load(f)
    n = page["n_fresh_queries"]
    one_hit = np.array([5.0] + [50.0] * (n - 1))  # one query under the threshold
    m, sd = output.threshold_rate(one_hit, page["nmse_threshold"])
    assert (round(m, 2), round(sd, 2)) == tuple(page["threshold_mean_sd_norot"])
    m, sd = output.threshold_rate(np.full(n, 2.0), page["nmse_threshold"])
    assert (round(m, 2), round(sd, 2)) == tuple(page["threshold_mean_sd_rot7"])
    # a 0/1 indicator's population sd is sqrt(m (1 - m))
    for hits in range(n + 1):
        x = np.array([1.0] * hits + [0.0] * (n - hits))
        m, sd = output.mean_popsd(x)
        assert abs(sd - np.sqrt(m * (1 - m))) < 1e-12
