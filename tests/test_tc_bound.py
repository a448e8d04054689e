"""The error bound the tensor-core cache write (dense R) charges, checked on the host
against an emulation of the worst-case accumulation it assumes (numpy, no GPU, no
product code).

Model: x (bf16) times R split exactly into three bf16 limbs; every product is exact;
each 16-product MMA adds its products to the accumulator one at a time, each add
aligning the smaller addend to the larger one's fp32 precision by truncation toward
zero and truncating the sum to 24 significant bits (the worst chunking the bound
allows for).  Four accumulators take K steps 2a and 2a + 1, limbs from lo to hi, and
are summed in fp32; the result must lie within 210 u ||x|| ||R_:,d|| of the exact x R
(u = 2^-24), the kernel's charge.  The charge is an a-priori worst case over every
chunking and sign pattern; on these inputs the emulated error is a few u ||x|| ||R||,
so the check pins the split and the MMA order (exact limbs, four accumulators) rather
than the constant's tightness."""
import numpy as np

from int2_kv_cache_gb300.workloads import learned_style_rotation, round_bf16

U = 2.0 ** -24


def _trunc24(v):
    """Truncate (toward zero) to 24 significant bits; v float64."""
    m, e = np.frexp(v)  # v = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.trunc(m * 2.0 ** 24) / 2.0 ** 24, e)


def _add_truncating(d, p):
    """d + p with the smaller addend truncated to the larger one's ulp, then the sum truncated."""
    big = np.maximum(np.abs(d), np.abs(p))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(big > 0, big, 1.0)))
    ulp = np.ldexp(1.0, (e - 23).astype(int))
    small_is_d = np.abs(d) < np.abs(p)
    dd = np.where(small_is_d, np.trunc(d / ulp) * ulp, d)
    pp = np.where(small_is_d, p, np.trunc(p / ulp) * ulp)
    return _trunc24(dd + pp)


def _limbs(r):
    hi = round_bf16(r)
    r1 = (r - hi).astype(np.float32)
    mid = round_bf16(r1)
    lo = round_bf16((r1 - mid).astype(np.float32))
    return [lo.astype(np.float64), mid.astype(np.float64), hi.astype(np.float64)]  # smallest first


def _emulate(x, r, n_acc):
    """x [n, 128] (bf16 values), r [128, 128] fp32 -> y [n, 128] under the model."""
    limbs = _limbs(r)
    steps = 8 // n_acc
    accs = []
    for a in range(n_acc):
        d = np.zeros((x.shape[0], r.shape[1]))
        for limb in limbs:
            for s in range(steps):
                k0 = 16 * (steps * a + s)
                for k in range(k0, k0 + 16):
                    d = _add_truncating(d, x[:, k:k + 1] * limb[k][None, :])  # exact products
        accs.append(d.astype(np.float32))
    y = accs[0]
    for t in accs[1:]:
        y = (y + t).astype(np.float32)
    return y.astype(np.float64)


def test_four_accumulators_stay_within_the_charge():
    rng = np.random.default_rng(20261202)
    r = learned_style_rotation(3, 0, 1)[0].astype(np.float32)
    x = rng.standard_normal((96, 128)).astype(np.float32)
    x[:, rng.choice(128, 6, replace=False)] += 10.0  # key-like outlier channels
    x = round_bf16(x).astype(np.float64)
    exact = x @ r.astype(np.float64)
    y = _emulate(x, r, 4)
    bound = 210 * U * np.linalg.norm(x, axis=1)[:, None] * np.linalg.norm(r.astype(np.float64), axis=0)[None, :]
    err = np.abs(y - exact)
    assert np.all(err <= bound), float((err / bound).max())
    # the emulation is not vacuous: the modelled error is a visible fraction of the charge
    assert (err / bound).max() > 1e-3
