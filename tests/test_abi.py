"""The C-ABI library loads, exports every entry point declared in include/kvq.h,
and its host-side validation rejects bad arguments before touching the GPU.
No kernel is launched here (these run without a GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

H = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def kvq():
    from int2_kv_cache_gb300 import _build
    _build.build()
    import int2_kv_cache_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(H).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvq):
    names = declared_functions()
    assert len(names) >= 12
    lib = kvq.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(kvq.EXPORTED) | {"kvq_last_error"}


def test_binding_names_match_c_names(kvq):
    for n in kvq.EXPORTED:
        if n in ("kvq_last_error",):
            continue
        assert callable(getattr(kvq, n)), n


def _layout(kvq, **kw):
    d = dict(page_tokens=16, n_kv_heads=8, n_q_heads=32, num_blocks=100, max_blocks_per_seq=10)
    d.update(kw)
    lay = kvq.make_layout(**d)
    return lay


def test_pool_bytes(kvq):
    lay = _layout(kvq, num_blocks=256, n_kv_heads=4, n_q_heads=4)
    assert kvq.kvq_pool_bytes(lay) == 256 * 4 * 1152
    lay8 = _layout(kvq, page_tokens=8, num_blocks=3, n_kv_heads=2, n_q_heads=2)
    assert kvq.kvq_pool_bytes(lay8) == 3 * 2 * 576


def _ws_bytes(n_seqs, hkv, gqa, n_ctas):
    """Documented decode workspace: partials [4 n_ctas + U][gqa][132] f32, query
    fragments [U][16 NT][32] u32, constants [U][gqa][4] f32, slice spans [U] int2,
    each region rounded up to 256 bytes (U = n_seqs * hkv units)."""
    a = lambda x: (x + 255) // 256 * 256
    u = n_seqs * hkv
    nt = (gqa + 3) // 4
    return (a((4 * n_ctas + u) * gqa * 132 * 4) + a(u * 16 * nt * 32 * 4) + a(u * gqa * 16) + a(u * 8))


def test_decode_workspace_size(kvq):
    lay = _layout(kvq)
    assert kvq.kvq_decode_workspace_size(lay, 16, 160, 5) == _ws_bytes(16, 8, 4, 5)
    # library's choice: one full wave (4 blocks per SM), capped at 16 chunks per block
    auto = kvq.kvq_decode_workspace_size(lay, 16, 160, 0)
    assert auto == _ws_bytes(16, 8, 4, (16 * 8 * 5 + 15) // 16)
    lay8 = _layout(kvq, n_q_heads=64, max_blocks_per_seq=4096)
    assert kvq.kvq_decode_workspace_size(lay8, 16, 32768, 0) == _ws_bytes(16, 8, 8, 3 * 152)
    assert kvq.kvq_decode_workspace_size(lay, 16, 160, 1) < kvq.kvq_decode_workspace_size(lay, 16, 160, 2)


def _status(kvq, fn, *args):
    return fn(*args)


def test_unsupported_head_dim_and_page_size(kvq):
    lib = kvq.lib()
    lay = _layout(kvq)
    lay.head_dim = 64
    out = ctypes.c_size_t(0)
    assert lib.kvq_decode_workspace_size(ctypes.byref(lay), 1, 16, 1, ctypes.byref(out)) == kvq.KVQ_EUNSUPPORTED
    assert b"head_dim" in lib.kvq_last_error()
    lay = _layout(kvq, page_tokens=32)
    assert lib.kvq_decode_workspace_size(ctypes.byref(lay), 1, 16, 1, ctypes.byref(out)) == kvq.KVQ_EUNSUPPORTED
    lay = _layout(kvq, n_q_heads=24)  # 3 query heads per KV head
    assert lib.kvq_decode_workspace_size(ctypes.byref(lay), 1, 16, 1, ctypes.byref(out)) == kvq.KVQ_EUNSUPPORTED
    lay = _layout(kvq, n_q_heads=12)  # not a multiple
    assert lib.kvq_decode_workspace_size(ctypes.byref(lay), 1, 16, 1, ctypes.byref(out)) == kvq.KVQ_EINVAL


def test_quantize_append_rejects_bad_arguments(kvq):
    lib = kvq.lib()
    lay = _layout(kvq)
    ident = kvq.KvqRot(0, None, None)
    fake = 0x10000  # aligned but never dereferenced: validation fails first
    # bad clip
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, fake, fake, 0, fake, fake, fake, ident, ident, None,
                                 1.5, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL and b"clip" in lib.kvq_last_error()
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, fake, fake, 0, fake, fake, fake, ident, ident, None,
                                 0.0, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL
    # null pointer
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, None, fake, 0, fake, fake, fake, ident, ident, None,
                                 1.0, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL and b"k is NULL" in lib.kvq_last_error()
    # misaligned pointer
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, fake + 4, fake, 0, fake, fake, fake, ident, ident, None,
                                 1.0, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL and b"aligned" in lib.kvq_last_error()
    # signed Hadamard without signs
    bad = kvq.KvqRot(1, None, None)
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, fake, fake, 0, fake, fake, fake, bad, ident, None,
                                 1.0, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL and b"signs" in lib.kvq_last_error()
    # unknown rotation kind / dtype
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, fake, fake, 0, fake, fake, fake, kvq.KvqRot(7, None, None),
                                 ident, None, 1.0, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 4, fake, fake, 5, fake, fake, fake, ident, ident, None,
                                 1.0, 1.0, fake, None)
    assert st == kvq.KVQ_EINVAL
    # nothing to do is OK without touching any pointer
    st = lib.kvq_quantize_append(ctypes.byref(lay), 1, 0, None, None, 0, None, None, None, ident, ident, None,
                                 1.0, 1.0, None, None)
    assert st == kvq.KVQ_OK


def test_decode_rejects_bad_arguments(kvq):
    lib = kvq.lib()
    lay = _layout(kvq)
    ident = kvq.KvqRot(0, None, None)
    fake = 0x10000
    # max_seq_len beyond the block table
    st = lib.kvq_decode_attention(ctypes.byref(lay), 1, fake, 0, fake, 161, fake, ident, fake, 1, fake, 1 << 20,
                                  fake, None)
    assert st == kvq.KVQ_EINVAL
    # workspace too small
    st = lib.kvq_decode_attention(ctypes.byref(lay), 2, fake, 0, fake, 160, fake, ident, fake, 4, fake, 16, fake, None)
    assert st == kvq.KVQ_EINVAL and b"workspace" in lib.kvq_last_error()
    # zero sequences is a no-op
    assert lib.kvq_decode_attention(ctypes.byref(lay), 0, None, 0, None, 0, None, ident, None, 0, None, 0, None,
                                    None) == kvq.KVQ_OK


def test_calib_rejects_bad_arguments(kvq):
    lib = kvq.lib()
    fake = 0x10000
    rots = (kvq.KvqRot * 1)(kvq.KvqRot(0, None, None))
    clips = (ctypes.c_float * 2)(1.0, 1.2)
    st = lib.kvq_calib_nmse(64, 4, 2, 2, 128, fake, fake, fake, 0, fake, 0, 1, rots, 2, clips, None, 0, fake, fake,
                            fake, 1 << 30, None)
    assert st == kvq.KVQ_EINVAL and b"clip" in lib.kvq_last_error()
    clips = (ctypes.c_float * 1)(1.0)
    st = lib.kvq_calib_nmse(20000, 4, 2, 2, 128, fake, fake, fake, 0, fake, 0, 1, rots, 1, clips, None, 0, fake, fake,
                            fake, 1 << 30, None)
    assert st == kvq.KVQ_EUNSUPPORTED
    out = ctypes.c_size_t(0)
    assert lib.kvq_calib_workspace_size(64, 65, 2, 2, 0, ctypes.byref(out)) == kvq.KVQ_EINVAL
    assert lib.kvq_calib_workspace_size(64, 4, 2, 2, 0, ctypes.byref(out)) == kvq.KVQ_OK and out.value > 0


def test_window_arguments_are_checked(kvq):
    lib = kvq.lib()
    lay = _layout(kvq)
    ident = kvq.KvqRot(0, None, None)
    fake = 0x10000

    def append(win, n_new=4):
        return lib.kvq_window_append(ctypes.byref(lay), 1, n_new, fake, fake, 0, fake, fake, None,
                                     ctypes.byref(win), None)

    assert append(kvq.KvqWindow(32, 8, fake)) == kvq.KVQ_EINVAL and b"sink" in lib.kvq_last_error()
    assert append(kvq.KvqWindow(64, 12, fake)) == kvq.KVQ_EINVAL and b"recent" in lib.kvq_last_error()
    assert append(kvq.KvqWindow(64, 8, None)) == kvq.KVQ_EINVAL and b"buf" in lib.kvq_last_error()
    assert append(kvq.KvqWindow(64, 8, fake + 8)) == kvq.KVQ_EINVAL
    assert append(kvq.KvqWindow(65536, 8, fake)) == kvq.KVQ_EUNSUPPORTED
    # no windows, or nothing to append: OK without touching a pointer
    assert append(kvq.KvqWindow(0, 0, None)) == kvq.KVQ_OK
    assert append(kvq.KvqWindow(64, 8, fake), n_new=0) == kvq.KVQ_OK


def test_windowed_workspace_adds_a_second_partial_set(kvq):
    lay = _layout(kvq, max_blocks_per_seq=4096)
    a = lambda x: (x + 255) // 256 * 256
    n_seqs, ctas = 16, 5
    plain = kvq.kvq_decode_workspace_size(lay, n_seqs, 160, ctas)
    assert kvq.kvq_decode_workspace_size_win(lay, n_seqs, 160, None, ctas) == plain
    assert kvq.kvq_decode_workspace_size_win(lay, n_seqs, 160, kvq.Window(0, 0), ctas) == plain
    u = n_seqs * 8
    win = kvq.Window(64, 256, None)
    win.buf = None
    # a window struct with sizes needs a buffer even for the size query
    with pytest.raises(kvq.KvqError):
        kvq.kvq_decode_workspace_size_win(lay, n_seqs, 160, win, ctas)

    class _Buf:  # an aligned address standing in for a device buffer (never dereferenced)
        def data_ptr(self):
            return 0x10000

    win.buf = _Buf()
    got = kvq.kvq_decode_workspace_size_win(lay, n_seqs, 160, win, ctas)
    extra = a((4 * ctas + u) * 4 * 132 * 4) + a(u * 16 * 1 * 32 * 4) + a(u * 8)
    assert got == plain + extra


def test_report_arguments_are_checked(kvq):
    lib = kvq.lib()
    fake = 0x10000
    ident = kvq.KvqRot(0, None, None)
    out = ctypes.c_size_t(0)
    assert lib.kvq_report_workspace_size(64, 65, 2, 2, ctypes.byref(out)) == kvq.KVQ_EINVAL
    assert lib.kvq_report_workspace_size(64, 4, 2, 2, ctypes.byref(out)) == kvq.KVQ_OK and out.value > 0
    # more positions than tokens, an unsupported head group, a bad clip, a misaligned mu
    args = lambda **kw: dict(dict(n_tok=64, n_qpos=4, hkv=2, gqa=2, d_model=128, clip_k=1.0, clip_v=1.0, mu=None), **kw)

    def call(a):
        return lib.kvq_head_error_report(a["n_tok"], a["n_qpos"], a["hkv"], a["gqa"], a["d_model"], fake, fake, fake,
                                         0, fake, 0, ident, ident, a["mu"], a["clip_k"], a["clip_v"], fake, fake,
                                         1 << 30, None)

    assert call(args(n_qpos=65)) == kvq.KVQ_EINVAL
    assert call(args(gqa=3)) == kvq.KVQ_EUNSUPPORTED
    assert call(args(clip_v=0.0)) == kvq.KVQ_EINVAL and b"clip" in lib.kvq_last_error()
    assert call(args(mu=fake + 4)) == kvq.KVQ_EINVAL and b"mu" in lib.kvq_last_error()
    assert call(args(n_tok=20000, n_qpos=4)) == kvq.KVQ_EUNSUPPORTED
