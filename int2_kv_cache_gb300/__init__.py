"""Python binding of libkvq (rotated INT2 KV-cache attention for GB300).

Argument marshalling only: every computation runs in the CUDA kernels of
``libkvq.so`` behind the C ABI declared in ``include/kvq.h``.  PyTorch supplies
device memory and streams.  There is no CPU path: if the library has not been
built, importing the binding functions raises.

Functions carry the C names (``kvq_quantize_append``, ``kvq_decode_attention``,
``kvq_out_proj``, ``kvq_calib_nmse`` and helpers) and take torch tensors.

A decode step, end to end (shapes as in ``include/kvq.h``)::

    import torch, int2_kv_cache_gb300 as kvq
    from int2_kv_cache_gb300 import _build
    _build.build()                                   # nvcc, sm_103a, in-tree libkvq.so
    lay = kvq.make_layout(page_tokens=16, n_kv_heads=8, n_q_heads=32, num_blocks=nb, max_blocks_per_seq=mb)
    pool = torch.zeros(kvq.kvq_pool_bytes(lay), dtype=torch.uint8, device="cuda")
    rk = kvq.DeviceRot("dense", dense=r_k)           # [H_kv, 128, 128] fp32; or "signed_hadamard" / "identity"
    rv = kvq.DeviceRot("dense", dense=r_v)
    kvq.kvq_key_mean(k_calib, mu)                    # Eq. 19; then mu R_K (Eq. 20):
    kvq.kvq_rotate_heads(mu[None], rk, mu_rot[None])
    kvq.kvq_quantize_append(lay, k, v, cu_new, start_pos, table, rk, rv, mu_rot, 0.96, 0.92, pool)
    ws = torch.empty(kvq.kvq_decode_workspace_size(lay, n_seqs, max_len), dtype=torch.uint8, device="cuda")
    kvq.kvq_decode_attention(lay, q, seq_lens, max_len, table, rk, pool, ws, o_rot)
    kvq.kvq_fold_wo(w_o, 32, 8, rv, w_fold)          # once: W_O R_V (Eqs. 29-31)
    kvq.kvq_out_proj(o_rot.reshape(n_seqs, -1), w_fold, y)

With BF16 sink / recent windows, add ``win = kvq.Window(64, 256, buf)`` (``buf`` of
``kvq.Window.buffer_bytes(n_seqs, 8, 64, 256)`` bytes), call ``kvq_window_append(lay,
k, v, cu_new, start_pos, mu, win)`` beside the append, and decode with
``kvq_decode_attention_win(lay, q, seq_lens, max_len, table, rk, rv, pool, win, ws, o_rot)``
(workspace from ``kvq_decode_workspace_size_win``).  Candidate selection:
``kvq_calib_nmse``; per-head error report: ``kvq_head_error_report``.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as LIB_PATH

KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_ECUDA, KVQ_EDEVICE_FLAG = 0, -1, -2, -3, -4
ROT_KIND = {"identity": 0, "signed_hadamard": 1, "dense": 2}
KVQ_F32, KVQ_BF16 = 0, 1
HEAD_DIM = 128


class KvqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"kvq status {status}: {message}")
        self.status = status


class KvqLayout(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("page_tokens", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int)]


class KvqRot(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("signs", ctypes.c_void_p), ("dense", ctypes.c_void_p)]


class KvqOptrTrace(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("n_tok", ctypes.c_int),
                ("n_qpos", ctypes.c_int)]


class KvqWindow(ctypes.Structure):
    _fields_ = [("sink_tokens", ctypes.c_int), ("recent_tokens", ctypes.c_int), ("buf", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libkvq.so (built in-tree by ``_build.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkvq.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, st, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
        lp = ctypes.POINTER(KvqLayout)
        wp = ctypes.POINTER(KvqWindow)
        tp = ctypes.POINTER(KvqOptrTrace)
        sigs = {
            "kvq_last_error": ([], ctypes.c_char_p),
            "kvq_pool_bytes": ([lp], sz),
            "kvq_device_check": ([vp], st),
            "kvq_key_mean": ([i, i, vp, i, vp, vp], st),
            "kvq_rotate_heads": ([i, i, i, vp, KvqRot, vp, vp], st),
            "kvq_quantize_append": ([lp, i, i, vp, vp, i, vp, vp, vp, KvqRot, KvqRot, vp, f, f, vp, vp], st),
            "kvq_decode_workspace_size": ([lp, i, i, i, ctypes.POINTER(sz)], st),
            "kvq_decode_attention": ([lp, i, vp, i, vp, i, vp, KvqRot, vp, i, vp, sz, vp, vp], st),
            "kvq_decode_attention_noalloc": ([lp, i, vp, i, vp, i, vp, KvqRot, vp, i, vp, vp], st),
            "kvq_decode_step": ([lp, i, vp, vp, vp, i, vp, i, vp, KvqRot, KvqRot, vp, f, f, vp, i, vp, sz, vp, vp],
                                st),
            "kvq_window_append": ([lp, i, i, vp, vp, i, vp, vp, vp, wp, vp], st),
            "kvq_decode_step_win": ([lp, i, vp, vp, vp, i, vp, i, vp, KvqRot, KvqRot, vp, vp, f, f, vp, wp, i, vp, sz,
                                     vp, vp], st),
            "kvq_decode_workspace_size_win": ([lp, i, i, i, wp, ctypes.POINTER(sz)], st),
            "kvq_decode_attention_win": ([lp, i, vp, i, vp, i, vp, KvqRot, KvqRot, vp, wp, i, vp, sz, vp, vp], st),
            "kvq_fold_wo": ([i, i, i, vp, i, KvqRot, vp, i, vp], st),
            "kvq_out_proj": ([i, i, i, vp, vp, i, vp, vp], st),
            "kvq_wo_packed_bytes": ([i, i, ctypes.POINTER(sz)], st),
            "kvq_pack_wo": ([i, i, vp, vp, vp], st),
            "kvq_out_proj_packed": ([i, i, i, vp, vp, vp, vp], st),
            "kvq_calib_workspace_size": ([i, i, i, i, i, ctypes.POINTER(sz)], st),
            "kvq_report_workspace_size": ([i, i, i, i, ctypes.POINTER(sz)], st),
            "kvq_head_error_report": ([i, i, i, i, i, vp, vp, vp, i, vp, i, KvqRot, KvqRot, vp, f, f, vp, vp, sz,
                                       vp], st),
            "kvq_calib_nmse": ([i, i, i, i, i, vp, vp, vp, i, vp, i, i, ctypes.POINTER(KvqRot), i,
                                ctypes.POINTER(ctypes.c_float), vp, i, vp, vp, vp, sz, vp], st),
            "kvq_optr_workspace_size": ([i, i, i, i, i, ctypes.POINTER(sz)], st),
            "kvq_optr_loss_grad": ([i, tp, i, i, vp, vp, vp, vp, vp, f, f, f, vp, vp, vp, sz, vp], st),
            "kvq_optr_calibrate_head": ([tp, tp, i, i, vp, vp, vp, vp, f, f, f, i, f, i, vp, vp, vp, vp, vp, sz,
                                         vp], st),
        }
        for name, (argtypes, restype) in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = argtypes
            fn.restype = restype
        _lib = L
    return _lib


EXPORTED = ("kvq_last_error", "kvq_pool_bytes", "kvq_device_check", "kvq_key_mean", "kvq_rotate_heads",
            "kvq_quantize_append", "kvq_decode_workspace_size", "kvq_decode_attention",
            "kvq_decode_attention_noalloc", "kvq_decode_step", "kvq_decode_step_win", "kvq_window_append", "kvq_decode_workspace_size_win",
            "kvq_decode_attention_win", "kvq_fold_wo",
            "kvq_out_proj", "kvq_wo_packed_bytes", "kvq_pack_wo", "kvq_out_proj_packed", "kvq_calib_workspace_size", "kvq_calib_nmse", "kvq_report_workspace_size",
            "kvq_head_error_report", "kvq_optr_workspace_size", "kvq_optr_loss_grad", "kvq_optr_calibrate_head")


def _check(status: int) -> None:
    if status != KVQ_OK:
        raise KvqError(status, lib().kvq_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return KVQ_F32
    if t.dtype == torch.bfloat16:
        return KVQ_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _contig(t, name):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class DeviceRot:
    """A rotation spec with its device tensors kept alive."""

    def __init__(self, kind: str, signs=None, dense=None):
        self.kind = kind
        self.signs = signs
        self.dense = dense

    @classmethod
    def from_spec(cls, rot, device="cuda"):
        import torch
        s = torch.as_tensor(rot.signs, dtype=torch.float32, device=device).contiguous() if rot.signs is not None else None
        d = torch.as_tensor(rot.dense, dtype=torch.float32, device=device).contiguous() if rot.dense is not None else None
        return cls(rot.kind, s, d)

    @property
    def c(self) -> KvqRot:
        return KvqRot(ROT_KIND[self.kind], _ptr(self.signs), _ptr(self.dense))


def make_layout(page_tokens: int, n_kv_heads: int, n_q_heads: int, num_blocks: int,
                max_blocks_per_seq: int) -> KvqLayout:
    return KvqLayout(HEAD_DIM, page_tokens, n_kv_heads, n_q_heads, num_blocks, max_blocks_per_seq)


def kvq_pool_bytes(layout: KvqLayout) -> int:
    return int(lib().kvq_pool_bytes(ctypes.byref(layout)))


def kvq_device_check(stream=None) -> None:
    _check(lib().kvq_device_check(_stream(stream)))


def kvq_key_mean(k, mu, stream=None) -> None:
    n_tok, h, d = k.shape
    _check(lib().kvq_key_mean(n_tok, h, _ptr(_contig(k, "k")), _dtype_code(k), _ptr(mu), _stream(stream)))


def kvq_rotate_heads(x, rot: DeviceRot, y, heads_per_rot: int = 1, stream=None) -> None:
    n_rows, n_heads, _ = x.shape
    _check(lib().kvq_rotate_heads(n_rows, n_heads, heads_per_rot, _ptr(_contig(x, "x")), rot.c, _ptr(y),
                                  _stream(stream)))


def kvq_quantize_append(layout: KvqLayout, k, v, cu_new, start_pos, block_table, rot_k: DeviceRot,
                        rot_v: DeviceRot, mu_rot_k, clip_k: float, clip_v: float, pool, stream=None) -> None:
    n_new = k.shape[0]
    n_seqs = start_pos.shape[0]
    _check(lib().kvq_quantize_append(ctypes.byref(layout), n_seqs, n_new, _ptr(_contig(k, "k")),
                                     _ptr(_contig(v, "v")), _dtype_code(k), _ptr(cu_new), _ptr(start_pos),
                                     _ptr(block_table), rot_k.c, rot_v.c, _ptr(mu_rot_k), clip_k, clip_v,
                                     _ptr(pool), _stream(stream)))


def kvq_decode_workspace_size(layout: KvqLayout, n_seqs: int, max_seq_len: int, n_splits: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvq_decode_workspace_size(ctypes.byref(layout), n_seqs, max_seq_len, n_splits, ctypes.byref(out)))
    return int(out.value)


def kvq_decode_attention(layout: KvqLayout, q, seq_lens, max_seq_len: int, block_table, rot_k: DeviceRot,
                         pool, workspace, o_rot, n_splits: int = 0, stream=None) -> None:
    n_seqs = q.shape[0]
    _check(lib().kvq_decode_attention(ctypes.byref(layout), n_seqs, _ptr(_contig(q, "q")), _dtype_code(q),
                                      _ptr(seq_lens), max_seq_len, _ptr(block_table), rot_k.c, _ptr(pool),
                                      n_splits, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _ptr(o_rot), _stream(stream)))


def kvq_decode_attention_noalloc(layout: KvqLayout, q, seq_lens, max_seq_len: int, block_table,
                                 rot_k: DeviceRot, pool, o_rot, n_splits: int = 0, stream=None) -> None:
    """Decode attention without a caller-provided workspace (for callers that may
    not allocate device memory); the split partials live in a fixed library buffer."""
    n_seqs = q.shape[0]
    _check(lib().kvq_decode_attention_noalloc(ctypes.byref(layout), n_seqs, _ptr(_contig(q, "q")), _dtype_code(q),
                                              _ptr(seq_lens), max_seq_len, _ptr(block_table), rot_k.c, _ptr(pool),
                                              n_splits, _ptr(o_rot), _stream(stream)))


def kvq_decode_step(layout: KvqLayout, q, k_new, v_new, seq_lens, max_seq_len: int, block_table,
                    rot_k: DeviceRot, rot_v: DeviceRot, mu_rot_k, clip_k: float, clip_v: float, pool, workspace,
                    o_rot, n_splits: int = 0, stream=None) -> None:
    """One decode step: each sequence's new token (k_new[b], v_new[b]) is appended at
    position seq_lens[b] - 1 and the decode attention reads it, in one call."""
    n_seqs = q.shape[0]
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise TypeError("q, k_new and v_new must share a dtype")
    _check(lib().kvq_decode_step(ctypes.byref(layout), n_seqs, _ptr(_contig(q, "q")), _ptr(_contig(k_new, "k_new")),
                                 _ptr(_contig(v_new, "v_new")), _dtype_code(q), _ptr(seq_lens), max_seq_len,
                                 _ptr(block_table), rot_k.c, rot_v.c, _ptr(mu_rot_k), clip_k, clip_v, _ptr(pool),
                                 n_splits, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(o_rot), _stream(stream)))


class Window:
    """BF16 sink / recent window sizes and the caller's record buffer (see kvq_window)."""

    def __init__(self, sink_tokens: int, recent_tokens: int, buf=None):
        self.sink_tokens = sink_tokens
        self.recent_tokens = recent_tokens
        self.buf = buf

    @staticmethod
    def buffer_bytes(n_seqs: int, n_kv_heads: int, sink_tokens: int, recent_tokens: int) -> int:
        return n_seqs * n_kv_heads * (sink_tokens + recent_tokens) * 512

    @property
    def c(self) -> KvqWindow:
        return KvqWindow(self.sink_tokens, self.recent_tokens, _ptr(self.buf))


def _win_ref(win):
    return None if win is None else ctypes.byref(win.c)


def kvq_window_append(layout: KvqLayout, k, v, cu_new, start_pos, mu_k, win: Window, stream=None) -> None:
    _check(lib().kvq_window_append(ctypes.byref(layout), start_pos.shape[0], k.shape[0], _ptr(_contig(k, "k")),
                                   _ptr(_contig(v, "v")), _dtype_code(k), _ptr(cu_new), _ptr(start_pos),
                                   _ptr(mu_k), _win_ref(win), _stream(stream)))


def kvq_decode_workspace_size_win(layout: KvqLayout, n_seqs: int, max_seq_len: int, win: Window | None,
                                  n_splits: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvq_decode_workspace_size_win(ctypes.byref(layout), n_seqs, max_seq_len, n_splits, _win_ref(win),
                                               ctypes.byref(out)))
    return int(out.value)


def kvq_decode_step_win(layout: KvqLayout, q, k_new, v_new, seq_lens, max_seq_len: int, block_table,
                        rot_k: DeviceRot, rot_v: DeviceRot, mu_rot_k, mu_k, clip_k: float, clip_v: float, pool,
                        win: Window | None, workspace, o_rot, n_splits: int = 0, stream=None) -> None:
    """kvq_decode_step with BF16 windows: the new token is also copied into its window
    slot (key centred by the unrotated mean mu_k) before the windowed decode reads it."""
    n_seqs = q.shape[0]
    if k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise TypeError("q, k_new and v_new must share a dtype")
    _check(lib().kvq_decode_step_win(ctypes.byref(layout), n_seqs, _ptr(_contig(q, "q")), _ptr(_contig(k_new, "k_new")),
                                     _ptr(_contig(v_new, "v_new")), _dtype_code(q), _ptr(seq_lens), max_seq_len,
                                     _ptr(block_table), rot_k.c, rot_v.c, _ptr(mu_rot_k), _ptr(mu_k), clip_k, clip_v,
                                     _ptr(pool), _win_ref(win), n_splits, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(o_rot), _stream(stream)))


def kvq_decode_attention_win(layout: KvqLayout, q, seq_lens, max_seq_len: int, block_table, rot_k: DeviceRot,
                             rot_v: DeviceRot, pool, win: Window | None, workspace, o_rot, n_splits: int = 0,
                             stream=None) -> None:
    n_seqs = q.shape[0]
    _check(lib().kvq_decode_attention_win(ctypes.byref(layout), n_seqs, _ptr(_contig(q, "q")), _dtype_code(q),
                                          _ptr(seq_lens), max_seq_len, _ptr(block_table), rot_k.c, rot_v.c,
                                          _ptr(pool),
                                          _win_ref(win), n_splits, _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(o_rot),
                                          _stream(stream)))


def kvq_fold_wo(w_o, n_q_heads: int, n_kv_heads: int, rot_v: DeviceRot, w_folded, stream=None) -> None:
    d_model = w_o.shape[0]
    _check(lib().kvq_fold_wo(d_model, n_q_heads, n_kv_heads, _ptr(_contig(w_o, "w_o")), _dtype_code(w_o),
                             rot_v.c, _ptr(w_folded), _dtype_code(w_folded), _stream(stream)))


def kvq_out_proj(x, w, y, stream=None) -> None:
    n_rows, k_dim = x.shape[0], x.numel() // max(1, x.shape[0])
    d_model = w.shape[0]
    _check(lib().kvq_out_proj(n_rows, d_model, k_dim, _ptr(_contig(x, "x")), _ptr(_contig(w, "w")),
                              _dtype_code(w), _ptr(y), _stream(stream)))


def kvq_calib_workspace_size(n_tok: int, n_qpos: int, n_kv_heads: int, gqa: int, joint: bool) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvq_calib_workspace_size(n_tok, n_qpos, n_kv_heads, gqa, int(joint), ctypes.byref(out)))
    return int(out.value)


def kvq_calib_nmse(q, k, v, w_o, cands, clips, mu, joint: bool, nmse, ref, workspace, stream=None) -> None:
    n_qpos, hq, _ = q.shape
    n_tok, hkv, _ = k.shape
    gqa = hq // hkv
    d_model = w_o.shape[0]
    rot_arr = (KvqRot * len(cands))(*[c.c for c in cands])
    clip_arr = (ctypes.c_float * len(clips))(*[float(c) for c in clips])
    _check(lib().kvq_calib_nmse(n_tok, n_qpos, hkv, gqa, d_model, _ptr(_contig(q, "q")), _ptr(_contig(k, "k")),
                                _ptr(_contig(v, "v")), _dtype_code(k), _ptr(_contig(w_o, "w_o")), _dtype_code(w_o),
                                len(cands), rot_arr, len(clips), clip_arr, _ptr(mu), int(joint), _ptr(nmse),
                                _ptr(ref), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)))


def kvq_report_workspace_size(n_tok: int, n_qpos: int, n_kv_heads: int, gqa: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvq_report_workspace_size(n_tok, n_qpos, n_kv_heads, gqa, ctypes.byref(out)))
    return int(out.value)


def kvq_head_error_report(q, k, v, w_o, rot_k: DeviceRot, rot_v: DeviceRot, mu, clip_k: float, clip_v: float, out,
                          workspace, stream=None) -> None:
    """out: float64 [5, H_kv] (E, E_key, E_val, E_naive, Y per KV head; see include/kvq.h)."""
    n_qpos, hq, _ = q.shape
    n_tok, hkv, _ = k.shape
    _check(lib().kvq_head_error_report(n_tok, n_qpos, hkv, hq // hkv, w_o.shape[0], _ptr(_contig(q, "q")),
                                       _ptr(_contig(k, "k")), _ptr(_contig(v, "v")), _dtype_code(k),
                                       _ptr(_contig(w_o, "w_o")), _dtype_code(w_o), rot_k.c, rot_v.c, _ptr(mu),
                                       float(clip_k), float(clip_v), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


# ---- OptR gradient calibration of one KV head ----
KVQ_OPTR_KEYS = 0
KVQ_OPTR_VALUES = 1


def _trace(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        _contig(t, name)
    return KvqOptrTrace(_ptr(q), _ptr(k), _ptr(v), k.shape[0], q.shape[0])


def kvq_optr_workspace_size(n_tok: int, n_qpos: int, gqa: int, n_tok_heldout: int = 0, n_qpos_heldout: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvq_optr_workspace_size(n_tok, n_qpos, n_tok_heldout, n_qpos_heldout, gqa, ctypes.byref(out)))
    return int(out.value)


def kvq_optr_loss_grad(phase: int, q, k, v, w_o, mu, r0, a, r_k_sel, clip_k: float, clip_v: float, lambda_k: float,
                       loss, grad, workspace, stream=None) -> None:
    """One OptR objective (keys: Eq. 14; values: Eq. 16) and dL/dA at R = r0 exp(a - a^T).
    q [n_qpos][gqa][128], k, v [n_tok][128], w_o [d_model][gqa*128], mu [128] (fp32);
    r0, a, r_k_sel, grad: fp64 [128][128]; loss: fp64 [1]."""
    tr = _trace(q, k, v)
    _check(lib().kvq_optr_loss_grad(phase, ctypes.byref(tr), q.shape[1], w_o.shape[0], _ptr(_contig(w_o, "w_o")),
                                    _ptr(mu), _ptr(r0), _ptr(a), _ptr(r_k_sel), clip_k, clip_v, lambda_k, _ptr(loss),
                                    _ptr(grad), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)))


def kvq_optr_calibrate_head(train, heldout, w_o, mu, r_k0, r_v0, clip_k: float, clip_v: float, lambda_k: float,
                            steps: int, lr: float, every: int, r_k, r_v, loss_k, loss_v, workspace,
                            stream=None) -> None:
    """Algorithm 1 for one KV head.  train / heldout: (q, k, v) tuples of fp32 tensors (heldout may be None)."""
    tr = _trace(*train)
    ho = _trace(*heldout) if heldout is not None else None
    q = train[0]
    _check(lib().kvq_optr_calibrate_head(ctypes.byref(tr), ctypes.byref(ho) if ho is not None else None, q.shape[1],
                                         w_o.shape[0], _ptr(_contig(w_o, "w_o")), _ptr(mu), _ptr(r_k0), _ptr(r_v0),
                                         clip_k, clip_v, lambda_k, steps, lr, every, _ptr(r_k), _ptr(r_v),
                                         _ptr(loss_k), _ptr(loss_v), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))


# ---- the folded W_O in the projection's box order ----
def kvq_wo_packed_bytes(d_model: int, k_dim: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().kvq_wo_packed_bytes(d_model, k_dim, ctypes.byref(out)))
    return int(out.value)


def kvq_pack_wo(w, w_packed, stream=None) -> None:
    """w: bf16 [d_model][k_dim] (e.g. kvq_fold_wo's output); w_packed: kvq_wo_packed_bytes bytes."""
    d_model, k_dim = w.shape
    _check(lib().kvq_pack_wo(d_model, k_dim, _ptr(_contig(w, "w")), _ptr(w_packed), _stream(stream)))


def kvq_out_proj_packed(x, w_packed, y, d_model: int, stream=None) -> None:
    n_rows, k_dim = x.shape
    _check(lib().kvq_out_proj_packed(n_rows, d_model, k_dim, _ptr(_contig(x, "x")), _ptr(w_packed), _ptr(y),
                                     _stream(stream)))
