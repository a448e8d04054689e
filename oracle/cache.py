"""The paged INT2 cache: record layout, write path and read path (fp64).

Test infrastructure only (see the package header).

Write path ("Output-Aware Rotation for INT2 KV-Cache Quantization", §4.1 and the
appendix paragraphs "Key-mean estimation and application" (Eqs. 19-20) and
"Rotated-query implementation" (Eq. 21)):

    mu_h          = mean over calibration tokens of the post-RoPE keys of head h   (Eq. 19)
    stored key    k_R = Q_2((k - mu_h) R_K,h ; c_K, 128)                          (Eq. 21)
    stored value  v_R = Q_2(v R_V,h ; c_V, 128)        (value path of Eq. 27: v' = v R_V)

The oracle centres before rotating, the plain form of Eq. 20; a kernel may
subtract the precomputed mu R instead (same value up to rounding).

Page layout (the pages say only that the cache is paged and that rotation keeps
its format; this layout is this implementation's choice): the pool is
[num_blocks][H_kv][record] bytes, one record per (physical page, KV head) of
72 * P bytes for P tokens per page:

    [0,    32P)  K codes, token slot o at 32*o (32 bytes = 128 two-bit codes)
    [32P,  64P)  V codes
    [64P,  68P)  K meta, slot o at 64P + 4*o: fp16 scale, then fp16 zero (little endian)
    [68P,  72P)  V meta

Token position pos of sequence b lives in physical page block_table[b][pos // P],
slot pos % P.

Pinned by tests/test_oracle_cache.py: hand-computed byte offsets on a tiny pool,
write/read round trips and the 1,048,576-byte payload of the evaluation page's
envelope.
"""
from __future__ import annotations

import numpy as np

from .quant import GROUP_BYTES, quantize_groups, pack_codes, unpack_codes, fp16_bits, fp16_from_bits

D = 128
META_BYTES = 4  # fp16 scale + fp16 zero


def record_bytes(page_tokens: int) -> int:
    return page_tokens * (2 * GROUP_BYTES + 2 * META_BYTES)


def pool_bytes(num_blocks: int, n_kv_heads: int, page_tokens: int) -> int:
    return num_blocks * n_kv_heads * record_bytes(page_tokens)


def offsets(page_tokens: int) -> dict:
    p = page_tokens
    return {"k_codes": 0, "v_codes": 32 * p, "k_meta": 64 * p, "v_meta": 68 * p}


def key_mean(k_cal: np.ndarray) -> np.ndarray:
    """Eq. 19: per-head, per-channel mean of post-RoPE calibration keys [N, H, 128] -> [H, 128]."""
    return np.asarray(k_cal, np.float64).mean(axis=0)


def rotate_heads(x: np.ndarray, r: np.ndarray, heads_per_rot: int = 1) -> np.ndarray:
    """x [..., n_heads, 128] -> x_h @ R_{h // heads_per_rot} for every head."""
    x = np.asarray(x, np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    for h in range(x.shape[-2]):
        out[..., h, :] = x[..., h, :] @ r[h // heads_per_rot]
    return out


def encode_tokens(k, v, r_k, r_v, mu, clip_k: float, clip_v: float, mu_rot=None) -> dict:
    """Quantize new tokens k, v [T, H, 128] for the cache (Eqs. 19-21, 27).

    The key is centred before rotation, x_K = (k - mu) R_K, or -- when ``mu_rot``
    (= mu R_K, [H, 128]) is given instead -- rotated then shifted,
    x_K = k R_K - mu R_K, the implementation form of Eq. 20.
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if mu_rot is not None:
        assert mu is None, "give mu or mu_rot, not both"
        xk = rotate_heads(k, r_k) - np.asarray(mu_rot, np.float64)[None]
    else:
        kc = k - (np.asarray(mu, np.float64)[None] if mu is not None else 0.0)
        xk = rotate_heads(kc, r_k)
    xv = rotate_heads(v, r_v)
    ck, sk, zk = quantize_groups(xk, clip_k)
    cv, sv, zv = quantize_groups(xv, clip_v)
    return {"xk": xk, "xv": xv, "ck": ck, "sk": sk, "zk": zk, "cv": cv, "sv": sv, "zv": zv}


def _meta_bytes(scale, zero) -> np.ndarray:
    m = np.stack([fp16_bits(scale), fp16_bits(zero)], axis=-1)  # [..., 2] uint16
    return np.ascontiguousarray(m).view(np.uint8).reshape(np.shape(scale) + (4,))


def write_tokens(pool: np.ndarray, n_kv_heads: int, page_tokens: int, table_row, start_pos: int,
                 enc: dict) -> None:
    """Append encoded tokens at positions start_pos.. of one sequence."""
    p = page_tokens
    rec = record_bytes(p)
    off = offsets(p)
    pool4 = pool.reshape(-1, n_kv_heads, rec)
    pk = pack_codes(enc["ck"])  # [T, H, 32]
    pv = pack_codes(enc["cv"])
    mk = _meta_bytes(enc["sk"], enc["zk"])  # [T, H, 4]
    mv = _meta_bytes(enc["sv"], enc["zv"])
    n = pk.shape[0]
    pos = start_pos + np.arange(n)
    blk = np.asarray(table_row, np.int64)[pos // p]  # physical page of every token
    assert np.all((blk >= 0) & (blk < pool4.shape[0]))
    slot = pos % p
    heads = np.arange(n_kv_heads)
    b3 = blk[:, None, None]
    h3 = heads[None, :, None]
    for base, width, data in ((off["k_codes"], 32, pk), (off["v_codes"], 32, pv),
                              (off["k_meta"], 4, mk), (off["v_meta"], 4, mv)):
        col = base + width * slot[:, None, None] + np.arange(width)[None, None, :]
        pool4[b3, h3, col] = data


def read_sequence(pool: np.ndarray, n_kv_heads: int, page_tokens: int, table_row, length: int) -> dict:
    """Codes and fp16 meta of positions 0..length-1 of one sequence."""
    p = page_tokens
    rec = record_bytes(p)
    off = offsets(p)
    pool4 = pool.reshape(-1, n_kv_heads, rec)
    n_pages = (length + p - 1) // p
    blocks = np.asarray(table_row[:n_pages], dtype=np.int64)
    recs = pool4[blocks]  # [n_pages, H, rec]

    def codes(base):
        b = recs[:, :, base: base + 32 * p].reshape(n_pages, n_kv_heads, p, 32)
        return unpack_codes(b.transpose(0, 2, 1, 3).reshape(n_pages * p, n_kv_heads, 32)[:length])

    def meta(base):
        m = recs[:, :, base: base + 4 * p].reshape(n_pages, n_kv_heads, p, 4)
        m = m.transpose(0, 2, 1, 3).reshape(n_pages * p, n_kv_heads, 4)[:length]
        m16 = np.ascontiguousarray(m).view(np.uint16)  # [L, H, 2]
        return fp16_from_bits(m16[..., 0]), fp16_from_bits(m16[..., 1])

    sk, zk = meta(off["k_meta"])
    sv, zv = meta(off["v_meta"])
    return {"ck": codes(off["k_codes"]), "sk": sk, "zk": zk,
            "cv": codes(off["v_codes"]), "sv": sv, "zv": zv}


def dequantized_sequence(pool, n_kv_heads, page_tokens, table_row, length):
    """k_R-hat, v_R-hat [L, H, 128] in the rotated basis (dequantized cache)."""
    r = read_sequence(pool, n_kv_heads, page_tokens, table_row, length)
    kh = r["zk"][..., None] + r["sk"][..., None] * r["ck"].astype(np.float64)
    vh = r["zv"][..., None] + r["sv"][..., None] * r["cv"].astype(np.float64)
    return kh, vh


def build_pool(case, r_k, r_v, mu=None, lengths=None, mu_rot=None, keep=False):
    """Encode every sequence of a workloads.DecodeCase into a fresh pool.

    Returns the pool, or (pool, per-sequence encodings) when ``keep``."""
    h = case.n_kv_heads
    p = case.page_tokens
    pool = np.zeros(pool_bytes(case.num_blocks, h, p), dtype=np.uint8)
    lengths = case.seq_lens if lengths is None else lengths
    encs = []
    for b in range(case.n_seqs):
        k, v = case.kv(b)
        n = int(lengths[b])
        enc = encode_tokens(k[:n], v[:n], r_k, r_v, mu, case.clip_k, case.clip_v, mu_rot=mu_rot)
        write_tokens(pool, h, p, case.block_table[b], 0, enc)
        if keep:
            encs.append(enc)
    return (pool, encs) if keep else pool
