"""BF16 sink and recent windows beside the INT2 cache (fp64).

Test infrastructure only (see the package header).

"Output-Aware Rotation for INT2 KV-Cache Quantization", §5 implementation
details and Table A (64 sink tokens and 256 recent tokens kept in BF16), §4.1
and the appendix paragraphs "OptR Algorithm" and "Key-mean estimation and
application" (window tokens skip INT2 quantization, their keys keep the same
centring, their values stay unchanged in BF16), Eqs. 24, 26 and 27 (the readout
in the rotated-V basis is o' = o R_V).

Readings (the pages leave these open):

* Window membership at length L: position p < L is a window token iff p < S
  (sink) or p >= L - R (recent); every other position is read from the INT2
  pages.  INT2 codes are still written for every token, so the pages do not
  depend on the windows.
* Window key  = bf16_rne(fp32(k - mu)): the centred, unrotated key, the
  difference taken in fp32 as a framework computes ``k.float() - mu`` and
  rounded once to bf16.  mu is the unrotated key mean (Eq. 19); no mu, no
  centring.  Its logit uses the unrotated query: q . k~ / sqrt(d), which equals
  (q R_K) . ((k - mu) R_K) / sqrt(d) up to the bf16 rounding (Eq. 24).
* Window value = bf16_rne(v): the value as given, unchanged (for bf16 inputs an
  exact copy).  The INT2 values are stored rotated (v R_V) and the readout is
  kept in the rotated-V basis (Eq. 27), so the window part of the readout is
  rotated once: o' = sum_INT2 p v^_R + (sum_window p v~) R_V.
* Storage, per (sequence, KV head): (S + R) / 8 records of 4,096 bytes, one
  record per 8 consecutive slots: the 8 keys, then the 8 values, each a row of
  128 bf16.  Position p lives in slot p (p < S) or S + (p mod R); slot s in
  record s // 8, row r = s % 8.  Inside a row, the 16-byte chunk c (channels
  8c .. 8c + 7) is stored at chunk position c XOR r.  (The XOR permutation is
  this implementation's choice; it lets a reader fetch the same chunk of the 8
  rows from 8 different shared-memory banks.)
* A recent-window copy is written only for tokens that are in the window at
  the sequence's new length (p >= start + n_new - R), so one append never
  writes a slot twice.  S must be a multiple of 64 and R a multiple of 8.

Pinned by tests/test_oracle_window.py: bf16 rounding against PyTorch's
float32 -> bfloat16 conversion, membership against a brute-force set, the record
layout as a bijection, ring contents after chunked appends, windowed decode with
empty windows equal to the plain decode, and lossless inputs on which the
windowed INT2 readout equals unquantized attention (Eqs. 1-2) exactly.
"""
from __future__ import annotations

import numpy as np

from .attention import rotate_queries, softmax

D = 128
RECORD_TOKENS = 8
ROW_BYTES = D * 2
RECORD_BYTES = 2 * RECORD_TOKENS * ROW_BYTES  # 4,096


def bf16_rne(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits, the
    exponent range of float32), ties to even; returns the rounded values."""
    x = np.asarray(x, np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e = np.frexp(xf)  # |x| = m 2^e, 0.5 <= m < 1
    # spacing of bf16 values around x: 2^(e - 8) for normal numbers, 2^-133 below 2^-126
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(xf / ulp) * ulp  # rint rounds half to even; both scalings are exact
    r[np.abs(r) > 3.3895313892515355e38] = np.inf  # beyond the largest finite bf16
    out[fin] = np.copysign(r, xf)
    return out


def bf16_bits(values) -> np.ndarray:
    """bfloat16 bit patterns of values that are exactly representable in bf16."""
    f = np.asarray(values, np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def check_window(sink: int, recent: int) -> None:
    assert sink >= 0 and recent >= 0 and sink % 64 == 0 and recent % RECORD_TOKENS == 0


def window_positions(length: int, sink: int, recent: int) -> np.ndarray:
    """Sorted positions p < length kept in BF16."""
    p = np.arange(length)
    return p[(p < sink) | (p >= length - recent)]


def int2_positions(length: int, sink: int, recent: int) -> np.ndarray:
    p = np.arange(length)
    return p[(p >= sink) & (p < length - recent)]


def slot_of(pos, sink: int, recent: int):
    pos = np.asarray(pos, np.int64)
    return np.where(pos < sink, pos, sink + pos % max(recent, 1))


def element_offset(slot, part: int, channel) -> np.ndarray:
    """Byte offset, inside one (sequence, KV head) window region, of channel
    ``channel`` of the key (part 0) or value (part 1) in ``slot``."""
    slot = np.asarray(slot, np.int64)
    channel = np.asarray(channel, np.int64)
    rec, r = slot // RECORD_TOKENS, slot % RECORD_TOKENS
    chunk = channel // 8
    return (rec * RECORD_BYTES + part * RECORD_TOKENS * ROW_BYTES + r * ROW_BYTES + ((chunk ^ r) * 16)
            + (channel % 8) * 2)


def region_bytes(sink: int, recent: int) -> int:
    return (sink + recent) // RECORD_TOKENS * RECORD_BYTES


def window_key(k, mu=None) -> np.ndarray:
    """bf16_rne(fp32(k - mu)) for k [..., H, 128] (fp32-representable) and mu [H, 128] or None."""
    k32 = np.asarray(k, np.float64).astype(np.float32)
    if mu is not None:
        k32 = k32 - np.asarray(mu, np.float64).astype(np.float32)  # one fp32 subtraction
    return bf16_rne(k32.astype(np.float64))


def window_value(v) -> np.ndarray:
    """bf16_rne(v) for v [..., H, 128]: the value unchanged, in bf16."""
    return bf16_rne(np.asarray(v, np.float64))


def write_window(region: np.ndarray, k, v, start_pos: int, sink: int, recent: int, mu) -> None:
    """Append tokens k, v [T, H, 128] of one sequence at positions start_pos..;
    region: uint8 [H, region_bytes(sink, recent)], written in place."""
    check_window(sink, recent)
    k = np.asarray(k, np.float64)
    n, h = k.shape[0], k.shape[1]
    new_len = start_pos + n
    kw = bf16_bits(window_key(k, mu))
    vw = bf16_bits(window_value(v))
    ch = np.arange(D)
    for t in range(n):
        p = start_pos + t
        if not (p < sink or p >= new_len - recent):
            continue
        s = int(slot_of(p, sink, recent))
        for part, src in ((0, kw), (1, vw)):
            off = element_offset(s, part, ch)
            for hh in range(h):
                b = src[t, hh].astype("<u2").view(np.uint8).reshape(D, 2)
                region[hh, off] = b[:, 0]
                region[hh, off + 1] = b[:, 1]


def read_window(region: np.ndarray, length: int, sink: int, recent: int):
    """Positions, keys and values [n, H, 128] (float64) of the window of a sequence of `length`."""
    pos = window_positions(length, sink, recent)
    h = region.shape[0]
    ch = np.arange(D)
    keys = np.empty((len(pos), h, D))
    vals = np.empty((len(pos), h, D))
    for i, p in enumerate(pos):
        s = int(slot_of(p, sink, recent))
        for part, dst in ((0, keys), (1, vals)):
            off = element_offset(s, part, ch)
            lo = region[:, off].astype(np.uint16)
            hi = region[:, off + 1].astype(np.uint16)
            dst[i] = bf16_from_bits(lo | (hi << 8))
    return pos, keys, vals


def decode_attention_windowed(q, k_hat, v_hat, win_pos, win_k, win_v, r_k, r_v, gqa: int, length: int,
                              sink: int, recent: int) -> np.ndarray:
    """One query per head over a sequence of `length` with BF16 windows.

    q [H_q, 128]; k_hat, v_hat [>= length, H_kv, 128]: the dequantized INT2
    cache in the rotated basis (only the INT2 positions are read);
    win_pos, win_k, win_v: ``read_window`` output (keys centred, values as
    given; neither rotated).  Returns o' [H_q, 128] in the rotated-V basis:
    the INT2 values are already rotated, the window values are rotated here.
    """
    q = np.asarray(q, np.float64)
    qr = rotate_queries(q, r_k, gqa)
    ipos = int2_positions(length, sink, recent)
    assert np.array_equal(np.sort(np.concatenate([ipos, win_pos])), np.arange(length))
    out = np.empty((q.shape[0], D))
    for j in range(q.shape[0]):
        h = j // gqa
        a = np.concatenate([k_hat[ipos, h, :] @ qr[j], win_k[:, h, :] @ q[j]]) / np.sqrt(D)
        p = softmax(a)
        n = len(ipos)
        out[j] = p[:n] @ v_hat[ipos, h, :] + (p[n:] @ win_v[:, h, :]) @ r_v[h]
    return out
