"""Group-wise asymmetric INT2 quantization Q_2(.; c, G) and its 2-bit packing (fp64).

Test infrastructure only (see the package header).

Source: "Output-Aware Rotation for INT2 KV-Cache Quantization", §3.1 (Eq. 4:
D_{R,c}(z) = Q_2(zR; c, G) R^T), the Implementation Details of §5 ("group-wise
affine INT2 quantization with a group size of 128" and clipping ratios), Table A,
and the 2.32 bits-per-element accounting (fp16 scale + fp16 zero per group of
128 two-bit codes).  The pages leave these steps open; the readings taken are:

* one group = the 128 channels of one token of one head (per-token groups, as
  the evaluation page's "per-token-group K/V quantization" states);
* clip ratio c scales both ends of the range: lo = c * min(x), hi = c * max(x);
* scale = fp16_rne((hi - lo) / 3), zero = fp16_rne(lo) -- zero is a float
  offset, not an integer zero point;
* code = clamp(round_half_even((x - zero) / scale), 0, 3) using the fp16-rounded
  scale and zero; a group with scale == 0 stores code 0 everywhere;
* dequantized value = zero + scale * code;
* packing: channel i of a group is stored in byte i // 4 at bits 2*(i % 4)
  (a group is 32 bytes).

Pinned by tests/test_oracle_quant.py: brute-force nearest-level search, a
hand-worked golden example, the grid invariant, the error bound, the identity
case of Eq. 4 and packing round trips.
"""
from __future__ import annotations

import numpy as np

G = 128
LEVELS = 4
GROUP_BYTES = G * 2 // 8  # 32


def fp16_rne(x) -> np.ndarray:
    """Round float64 values to the nearest IEEE binary16 (ties to even), as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def fp16_bits(x) -> np.ndarray:
    """IEEE binary16 bit patterns of values that are exactly representable in fp16."""
    h = np.asarray(x, dtype=np.float64).astype(np.float16)
    assert np.array_equal(h.astype(np.float64), np.asarray(x, dtype=np.float64)), "value not fp16-exact"
    return h.view(np.uint16)


def fp16_from_bits(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def quantize_groups(x: np.ndarray, clip: float):
    """Q_2 on groups along the last axis (length 128).

    Returns (codes uint8 in 0..3, scale, zero) where scale and zero are the
    fp16-rounded values (as float64), one per group.
    """
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] == G
    c = np.float64(clip)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    lo = c * mn
    hi = c * mx
    scale = fp16_rne((hi - lo) / 3.0)
    zero = fp16_rne(lo)
    s = scale[..., None]
    z = zero[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(s > 0, (x - z) / np.where(s > 0, s, 1.0), 0.0)
    codes = np.clip(np.rint(t), 0, LEVELS - 1).astype(np.uint8)
    return codes, scale, zero


def dequantize_groups(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    return (np.asarray(zero, np.float64)[..., None]
            + np.asarray(scale, np.float64)[..., None] * codes.astype(np.float64))


def quant_dequant(x: np.ndarray, clip: float) -> np.ndarray:
    """Q_2(x; c, 128): quantize then dequantize."""
    codes, s, z = quantize_groups(x, clip)
    return dequantize_groups(codes, s, z)


def rotated_quant_dequant(x: np.ndarray, r: np.ndarray, clip: float) -> np.ndarray:
    """D_{R,c}(x) = Q_2(x R; c, G) R^T (Eq. 4) for row vectors x [..., 128]."""
    return quant_dequant(np.asarray(x, np.float64) @ r, clip) @ r.T


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[..., 128] codes in 0..3 -> [..., 32] bytes; channel i -> byte i//4, bits 2*(i%4)."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] == G and codes.max(initial=0) < LEVELS
    c4 = codes.reshape(codes.shape[:-1] + (GROUP_BYTES, 4)).astype(np.uint32)
    b = c4[..., 0] | (c4[..., 1] << 2) | (c4[..., 2] << 4) | (c4[..., 3] << 6)
    return b.astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    assert packed.shape[-1] == GROUP_BYTES
    out = np.empty(packed.shape[:-1] + (GROUP_BYTES, 4), dtype=np.uint8)
    for i in range(4):
        out[..., i] = (packed >> (2 * i)) & 3
    return out.reshape(packed.shape[:-1] + (G,))


def near_boundary(x: np.ndarray, scale: np.ndarray, zero: np.ndarray, rel: float = 1e-6) -> np.ndarray:
    """Elements whose code could legitimately differ between two correct
    implementations that compute x in different floating-point precisions:
    |x - (zero + m*scale)| <= rel * max(|x|, scale) for a rounding midpoint
    m in {0.5, 1.5, 2.5}."""
    x = np.asarray(x, np.float64)
    s = np.asarray(scale, np.float64)[..., None]
    z = np.asarray(zero, np.float64)[..., None]
    tol = rel * np.maximum(np.abs(x), s)
    hit = np.zeros(x.shape, dtype=bool)
    for m in (0.5, 1.5, 2.5):
        hit |= np.abs(x - (z + m * s)) <= tol
    return hit


def group_near_fp16_tie(x: np.ndarray, clip: float, rel: float = 1e-6) -> np.ndarray:
    """Groups whose fp16 scale or zero sits within ``rel`` (relative) of an fp16
    rounding midpoint: another correct implementation may round them the other way."""
    x = np.asarray(x, np.float64)
    c = np.float64(clip)
    lo = c * x.min(axis=-1)
    hi = c * x.max(axis=-1)
    out = np.zeros(lo.shape, dtype=bool)
    for v in ((hi - lo) / 3.0, lo):
        r16 = np.asarray(v, np.float64).astype(np.float16)
        r = r16.astype(np.float64)
        up = np.nextafter(r16, np.float16(np.inf)).astype(np.float64)
        dn = np.nextafter(r16, np.float16(-np.inf)).astype(np.float64)
        for mid in ((r + up) / 2, (r + dn) / 2):
            out |= np.abs(v - mid) <= rel * np.abs(v)
    return out
