"""Pins for oracle.report: the per-head error report against the (separately
pinned) calibration sweep where the two coincide, the Eq. 8 split on inputs
where one side is stored losslessly, and pure-Python loops on a tiny case."""
import math

import numpy as np

from oracle import calib, report, rotations

D = 128


def _case(seed, n_tok=96, n_qpos=8, hkv=2, gqa=1, d_model=48):
    g = np.random.default_rng(seed)
    q = g.standard_normal((n_qpos, hkv * gqa, D))
    k = g.standard_normal((n_tok, hkv, D)) * 2.0
    k[..., :4] += 8.0
    v = g.standard_normal((n_tok, hkv, D))
    w = g.standard_normal((d_model, hkv * gqa * D)) / np.sqrt(hkv * gqa * D)
    r = np.stack([rotations.expm_skew(g.normal(0, 0.05, (D, D))) for _ in range(hkv)])
    mu = k.mean(axis=0)
    return q, k, v, w, r, mu


def test_one_query_head_per_kv_head_equals_the_calibration_sweep():
    q, k, v, w, r, mu = _case(1, gqa=1)
    rep = report.head_error_report(q, k, v, w, r, r, mu, 0.95, 0.95, 1)
    _, err, ref = calib.calib_sweep(q, k, v, w, [r], [0.95], mu, 1, False)
    assert np.allclose(rep["e"], err[0, 0], rtol=1e-12)
    assert np.allclose(rep["y"], ref, rtol=1e-12)
    eye = np.broadcast_to(np.eye(D), r.shape)
    _, err0, _ = calib.calib_sweep(q, k, v, w, [eye], [0.95], None, 1, False)
    assert np.allclose(rep["e_naive"], err0[0, 0], rtol=1e-12)


def test_identity_candidate_is_one_hundred_percent_of_naive():
    q, k, v, w, r, mu = _case(2, gqa=2)
    eye = np.broadcast_to(np.eye(D), r.shape)
    rep = report.head_error_report(q, k, v, w, eye, eye, None, 0.9, 0.92, 2)
    assert np.array_equal(rep["e"], rep["e_naive"]) and np.allclose(rep["rms_pct_of_naive"], 100.0)


def _on_grid(g, shape):
    lo = g.integers(-24, 0, shape[:-1] + (1,)) / 8.0
    s = g.integers(1, 12, shape[:-1] + (1,)) / 8.0
    i = g.integers(0, 4, shape)
    i[..., 0], i[..., 1] = 0, 3
    return lo + s * i


def test_eq8_split_when_one_side_is_lossless():
    """Keys on the INT2 grid (identity R_K, no centring): the key-induced term vanishes
    and the whole error is value-induced; and the other way round."""
    g = np.random.default_rng(3)
    n_tok, n_qpos, hkv, gqa = 80, 6, 2, 2
    q = g.standard_normal((n_qpos, hkv * gqa, D))
    w = g.standard_normal((32, hkv * gqa * D)) / 16
    eye = np.broadcast_to(np.eye(D), (hkv, D, D))
    exact = _on_grid(g, (n_tok, hkv, D))
    lossy = g.standard_normal((n_tok, hkv, D))
    rep = report.head_error_report(q, exact, lossy, w, eye, eye, None, 1.0, 1.0, gqa)
    assert np.all(rep["e_key"] < 1e-24 * rep["y"]) and np.allclose(rep["e"], rep["e_val"], rtol=1e-12)
    assert np.all(rep["e_val"] > 0)
    rep = report.head_error_report(q, lossy, exact, w, eye, eye, None, 1.0, 1.0, gqa)
    assert np.all(rep["e_val"] < 1e-24 * rep["y"]) and np.allclose(rep["e"], rep["e_key"], rtol=1e-12)
    assert np.all(rep["e_key"] > 0)


def test_split_terms_bound_the_total():
    q, k, v, w, r, mu = _case(4, gqa=4, hkv=1)
    rep = report.head_error_report(q, k, v, w, r, r, mu, 0.96, 0.92, 4)
    lo = (np.sqrt(rep["e_key"]) - np.sqrt(rep["e_val"])) ** 2
    hi = (np.sqrt(rep["e_key"]) + np.sqrt(rep["e_val"])) ** 2
    assert np.all(lo <= rep["e"] * (1 + 1e-12)) and np.all(rep["e"] <= hi * (1 + 1e-12))


def test_matches_pure_python_loops():
    g = np.random.default_rng(5)
    n_tok, n_qpos, hkv, gqa, dm = 6, 2, 1, 2, 3
    q = g.standard_normal((n_qpos, gqa, D))
    k = g.standard_normal((n_tok, hkv, D)) * 2
    v = g.standard_normal((n_tok, hkv, D))
    w = g.standard_normal((dm, gqa * D)) / 10
    r_k = rotations.expm_skew(g.normal(0, 0.2, (D, D)))[None]
    r_v = rotations.expm_skew(g.normal(0, 0.2, (D, D)))[None]
    mu = g.standard_normal((hkv, D))
    rep = report.head_error_report(q, k, v, w, r_k, r_v, mu, 0.9, 0.8, gqa)

    from oracle.quant import quant_dequant
    xk = quant_dequant(np.einsum("tc,cd->td", k[:, 0] - mu[0], r_k[0]), 0.9)  # effective rotated keys
    vq = quant_dequant(np.einsum("tc,cd->td", v[:, 0], r_v[0]), 0.8)
    v_eff = [[sum(vq[s][d] * r_v[0][c][d] for d in range(D)) for c in range(D)] for s in range(n_tok)]
    e = ek = ev = 0.0
    for i in range(n_qpos):
        t = n_tok - n_qpos + i
        for j in range(gqa):
            qj = q[i][j].tolist()
            qr = [sum(qj[c] * r_k[0][c][d] for c in range(D)) for d in range(D)]
            a = [sum(qj[c] * k[s][0][c] for c in range(D)) / math.sqrt(D) for s in range(t + 1)]
            at = [sum(qr[d] * xk[s][d] for d in range(D)) / math.sqrt(D) for s in range(t + 1)]
            p = [math.exp(x - max(a)) for x in a]
            p = [x / sum(p) for x in p]
            pt = [math.exp(x - max(at)) for x in at]
            pt = [x / sum(pt) for x in pt]
            for n in range(dm):
                wrow = w[n, j * D:(j + 1) * D].tolist()
                y = sum(p[s] * sum(v[s][0][c] * wrow[c] for c in range(D)) for s in range(t + 1))
                yt = sum(pt[s] * sum(v_eff[s][c] * wrow[c] for c in range(D)) for s in range(t + 1))
                yk = sum((pt[s] - p[s]) * sum(v[s][0][c] * wrow[c] for c in range(D)) for s in range(t + 1))
                yv = sum(pt[s] * sum((v_eff[s][c] - v[s][0][c]) * wrow[c] for c in range(D)) for s in range(t + 1))
                e += (yt - y) ** 2
                ek += yk ** 2
                ev += yv ** 2
    assert abs(rep["e"][0] - e) < 1e-10 * e
    assert abs(rep["e_key"][0] - ek) < 1e-10 * ek
    assert abs(rep["e_val"][0] - ev) < 1e-10 * ev
