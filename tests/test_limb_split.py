"""The arithmetic facts the tensor-core cache write (dense R) rests on, checked on
the host with numpy (no GPU, no product code): every fp32 value splits exactly into
three bf16 limbs by rounding to nearest, hi = bf16(x), mid = bf16(x - hi),
lo = x - hi - mid (so lo needs no rounding), fp32 (lo + mid) + hi gives x back, and
|mid| <= 2^-8 |x|, |lo| <= 2^-17 |x| (the sizes the MMA error bound charges), for
|x| >= 2^-100; below that the last limb reaches the fp32 subnormals and the split is
off by at most 2^-134 (half the smallest bf16 subnormal), which the kernel's absolute
error term covers."""
import numpy as np

from int2_kv_cache_gb300.workloads import round_bf16


def _values():
    rng = np.random.default_rng(20261202)
    x = np.concatenate([
        (rng.standard_normal(400_000) * s).astype(np.float32) for s in (1e-30, 1e-6, 1e-3, 0.088, 1.0, 1e3, 1e30)
    ])
    # values next to powers of two and bf16 rounding midpoints, where the carries happen
    p2 = np.float32(2.0) ** np.arange(-60, 60, dtype=np.float32)
    near = np.concatenate([np.nextafter(p2, np.float32(0)), np.nextafter(p2, np.float32(np.inf)),
                           p2 * np.float32(1 + 2.0 ** -8), p2 * np.float32(1 + 2.0 ** -8 + 2.0 ** -23),
                           p2 * np.float32(1 + 2.0 ** -8 - 2.0 ** -23)])
    u = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    raw = u.view(np.float32)
    raw = raw[np.isfinite(raw) & (np.abs(raw) > np.float32(1e-34)) & (np.abs(raw) < np.float32(1e34))]
    return np.concatenate([x, near, -near, raw]).astype(np.float32)


def test_three_bf16_limbs_hold_fp32_exactly():
    x = _values()
    x = x[np.abs(x) >= np.float32(2.0 ** -100)]
    assert x.size > 2_500_000
    hi = round_bf16(x)
    r1 = (x - hi).astype(np.float32)
    mid = round_bf16(r1)
    r2 = (r1 - mid).astype(np.float32)
    lo = round_bf16(r2)
    assert np.array_equal(lo, r2)  # the last limb needs no rounding
    assert np.array_equal(hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64), x.astype(np.float64))
    assert np.array_equal(((lo + mid).astype(np.float32) + hi).astype(np.float32), x)
    ax = np.abs(x.astype(np.float64))
    assert np.all(np.abs(mid.astype(np.float64)) <= 2.0 ** -8 * ax)
    assert np.all(np.abs(lo.astype(np.float64)) <= 2.0 ** -17 * ax)


def test_split_error_below_the_normal_range_is_tiny():
    x = _values()
    x = x[np.abs(x) < np.float32(2.0 ** -100)]
    hi = round_bf16(x)
    r1 = (x - hi).astype(np.float32)
    mid = round_bf16(r1)
    lo = round_bf16((r1 - mid).astype(np.float32))
    err = np.abs(hi.astype(np.float64) + mid + lo - x.astype(np.float64))
    assert err.max() <= 2.0 ** -134


def test_bf16_products_are_exact_in_fp32():
    rng = np.random.default_rng(7)
    a = round_bf16(rng.standard_normal(100_000).astype(np.float32) * 3)
    b = round_bf16(rng.standard_normal(100_000).astype(np.float32) * 1e-3)
    assert np.array_equal((a * b).astype(np.float64), a.astype(np.float64) * b.astype(np.float64))
