"""Shared plumbing for the GPU parity tests: upload seeded inputs, run the C-ABI
path, and compare against the fp64 oracle with the tolerances of the method's
parity rules:

* packed codes bit-exact, except elements within 1e-6 (relative) of a rounding
  boundary and whole groups whose fp16 scale/zero sit within 1e-6 of an fp16
  rounding midpoint; such mismatches are reported and must number <= 1e-5 of
  all elements (rounded up to a whole element);
* attention and post-W_O outputs: max |gpu - ref| / max |ref| <= 2e-3, over the
  whole tensor and within every output vector (one query head's readout, one row of y);
* NMSE: relative error <= 1e-4.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

CODE_EXEMPT_FRACTION = 1e-5
OUT_TOL = 2e-3
NMSE_TOL = 1e-4


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def kvq_lib():
    from int2_kv_cache_gb300 import _build
    _build.build()
    import int2_kv_cache_gb300 as kvq
    kvq.lib()
    return kvq


def dev(x, dtype: str = "f32"):
    """numpy float32 -> CUDA tensor (bf16 conversion is exact: values are bf16-exact)."""
    torch = torch_cuda()
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def dev_i32(x):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def normwise_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))


def rowwise_err(got, ref) -> float:
    """The same ratio per output vector (last axis: one query head's readout, one
    row of y): max over vectors of max |gpu - ref| / max |ref| within the vector,
    so a vector of small magnitude is held to its own size.  All-zero reference
    vectors must be matched exactly."""
    got = np.asarray(got, np.float64).reshape(-1, np.shape(got)[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, np.shape(ref)[-1])
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    if np.any((den == 0) & (num > 0)):
        return float("inf")
    nz = den > 0
    return float((num[nz] / den[nz]).max()) if nz.any() else 0.0


def out_err(got, ref) -> float:
    """Attention / post-W_O output error: the larger of the tensor-wise and the
    per-vector ratios (both are held to OUT_TOL)."""
    return max(normwise_err(got, ref), rowwise_err(got, ref))


# ---- reading a pool (test-side reader, independent of the oracle's) ----

def _records(pool: np.ndarray, h: int, p: int) -> np.ndarray:
    return np.asarray(pool, np.uint8).reshape(-1, h, 72 * p)


def seq_codes_meta(pool, h, p, table_row, length, which: str):
    """codes [L, H, 128] uint8 and meta bits [L, H, 2] uint16 of one sequence's K or V."""
    rec = _records(pool, h, p)
    n_pages = (length + p - 1) // p
    r = rec[np.asarray(table_row[:n_pages], np.int64)]  # [pages, H, 72p]
    c0 = 0 if which == "k" else 32 * p
    m0 = 64 * p if which == "k" else 68 * p
    cb = r[:, :, c0:c0 + 32 * p].reshape(n_pages, h, p, 32).transpose(0, 2, 1, 3).reshape(-1, h, 32)[:length]
    codes = np.stack([(cb >> (2 * i)) & 3 for i in range(4)], axis=-1).reshape(length, h, 128)
    mb = r[:, :, m0:m0 + 4 * p].reshape(n_pages, h, p, 4).transpose(0, 2, 1, 3).reshape(-1, h, 4)[:length]
    meta = np.ascontiguousarray(mb).view(np.uint16).reshape(length, h, 2)
    return codes.astype(np.uint8), meta


def compare_codes(gpu_pool, ora_pool, h, p, table, lengths, encs, clips, label="") -> dict:
    """Compare packed codes and meta of every sequence; enforce the exemption rules.

    encs: per-sequence oracle encodings (with the fp64 pre-quantization values xk, xv)."""
    from oracle import quant

    stats = {"elements": 0, "mismatch": 0, "meta_mismatch_groups": 0, "exempt_groups": 0}
    for b, length in enumerate(lengths):
        if length == 0:
            continue
        for which, clip in (("k", clips[0]), ("v", clips[1])):
            cg, mg = seq_codes_meta(gpu_pool, h, p, table[b], length, which)
            co, mo = seq_codes_meta(ora_pool, h, p, table[b], length, which)
            x = encs[b]["x" + which]
            s = encs[b]["s" + which]
            z = encs[b]["z" + which]
            group_ok = quant.group_near_fp16_tie(x, clip)
            elem_ok = quant.near_boundary(x, s, z) | group_ok[..., None]
            meta_bad = np.any(mg != mo, axis=-1)
            assert not np.any(meta_bad & ~group_ok), (
                f"{label} seq {b} {which}: fp16 meta differs in a group that is not at an fp16 tie "
                f"({int((meta_bad & ~group_ok).sum())} groups)")
            bad = cg != co
            assert not np.any(bad & ~elem_ok), (
                f"{label} seq {b} {which}: {int((bad & ~elem_ok).sum())} code(s) differ away from a rounding boundary")
            stats["elements"] += cg.size
            stats["mismatch"] += int(bad.sum())
            stats["meta_mismatch_groups"] += int(meta_bad.sum())
            stats["exempt_groups"] += int(group_ok.sum())
    limit = math.ceil(CODE_EXEMPT_FRACTION * stats["elements"])
    assert stats["mismatch"] <= limit, f"{label}: {stats['mismatch']} boundary mismatches > {limit}"
    return stats


class GpuCase:
    """A DecodeCase uploaded to the GPU, with the oracle's rotations and key shift."""

    def __init__(self, case, lengths=None, mu_mode: str = "cal"):
        import oracle
        self.kvq = kvq_lib()
        self.torch = torch_cuda()
        self.case = case
        self.lengths = np.asarray(case.seq_lens if lengths is None else lengths, np.int64)
        self.r_k = oracle.rotations.rot_matrices(case.rot_k, case.n_kv_heads)
        self.r_v = oracle.rotations.rot_matrices(case.rot_v, case.n_kv_heads)
        if mu_mode == "cal":
            mu = oracle.cache.key_mean(case.calibration_keys())
            self.mu_rot = np.einsum("hc,hcd->hd", mu, self.r_k).astype(np.float32)
        else:
            self.mu_rot = None
        self.layout = self.kvq.make_layout(case.page_tokens, case.n_kv_heads, case.n_q_heads, case.num_blocks,
                                           case.block_table.shape[1])
        self.table = dev_i32(case.block_table)
        self.rot_k = self.kvq.DeviceRot.from_spec(case.rot_k)
        self.rot_v = self.kvq.DeviceRot.from_spec(case.rot_v)
        self.mu_rot_dev = dev(self.mu_rot) if self.mu_rot is not None else None

    def new_pool(self):
        return self.torch.zeros(self.kvq.kvq_pool_bytes(self.layout), dtype=self.torch.uint8, device="cuda")

    def gpu_append_all(self, pool, chunks: int = 1):
        """Append every sequence's tokens with kvq_quantize_append (in `chunks` calls)."""
        c = self.case
        kv = [c.kv(b) for b in range(c.n_seqs)]
        bounds = [np.linspace(0, n, chunks + 1).round().astype(int) for n in self.lengths]
        for ci in range(chunks):
            ks, vs, cu, start = [], [], [0], []
            for b in range(c.n_seqs):
                lo, hi = bounds[b][ci], bounds[b][ci + 1]
                ks.append(kv[b][0][lo:hi])
                vs.append(kv[b][1][lo:hi])
                cu.append(cu[-1] + (hi - lo))
                start.append(lo)
            k = np.concatenate(ks) if ks else np.zeros((0, c.n_kv_heads, 128), np.float32)
            v = np.concatenate(vs)
            self.kvq.kvq_quantize_append(self.layout, dev(k, c.dtype), dev(v, c.dtype), dev_i32(cu), dev_i32(start),
                                         self.table, self.rot_k, self.rot_v, self.mu_rot_dev, c.clip_k, c.clip_v,
                                         pool)
        self.torch.cuda.synchronize()

    def oracle_pool(self):
        import oracle
        return oracle.cache.build_pool(self.case, self.r_k, self.r_v, None, lengths=self.lengths,
                                       mu_rot=self.mu_rot, keep=True)

    def gpu_decode(self, pool, q, n_splits=0, q_dtype=None):
        kvq = self.kvq
        c = self.case
        max_len = int(self.lengths.max()) if len(self.lengths) else 0
        ws_bytes = kvq.kvq_decode_workspace_size(self.layout, c.n_seqs, max_len, n_splits)
        ws = self.torch.empty(max(ws_bytes, 16), dtype=self.torch.uint8, device="cuda")
        out = self.torch.full((c.n_seqs, c.n_q_heads, 128), float("nan"), device="cuda")
        kvq.kvq_decode_attention(self.layout, dev(q, q_dtype or c.dtype), dev_i32(self.lengths), max_len,
                                 self.table, self.rot_k, pool, ws, out, n_splits=n_splits)
        self.torch.cuda.synchronize()
        return out.cpu().numpy()

    def oracle_decode(self, ora_pool, q, seqs=None):
        import oracle
        c = self.case
        out = {}
        for b in (range(c.n_seqs) if seqs is None else seqs):
            n = int(self.lengths[b])
            if n == 0:
                out[b] = np.zeros((c.n_q_heads, 128))
                continue
            kh, vh = oracle.cache.dequantized_sequence(ora_pool, c.n_kv_heads, c.page_tokens, c.block_table[b], n)
            out[b] = oracle.attention.decode_attention(q[b], kh, vh, self.r_k, c.gqa)
        return out


def assert_nmse_close(got, ref, label=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.abs(got - ref) / np.abs(ref)
    i = np.unravel_index(np.argmax(rel), rel.shape)
    assert rel.max() <= NMSE_TOL, f"{label}: worst NMSE rel err {rel.max():.3g} at {i}: gpu {got[i]} oracle {ref[i]}"
    return float(rel.max())
