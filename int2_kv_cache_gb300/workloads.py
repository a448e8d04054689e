"""Seeded synthetic inputs for rotated INT2 KV-cache attention.

This module only *draws* tensors: queries, post-RoPE keys, values, rotation
generators and sign vectors, output-projection weights, block tables and
context lengths.  It performs none of the method's arithmetic (no centring,
rotation of data, quantization, attention or projection).  Both the CUDA path
and the fp64 oracle consume exactly the arrays produced here, so the two share
inputs but no computation.

Shapes and statistics follow the workloads described in "Output-Aware Rotation
for INT2 KV-Cache Quantization" (OptR): head dimension 128, grouped-query
attention, keys with a few large per-channel offsets (the outlier channels of
its Figure 2), and the "Output-aware INT2 KV-cache rotation evaluation" page's
envelope (4,096 cached tokens x 4 KV heads, identity + 8 signed-Hadamard
candidates x 5 clip ratios).  The real traces (GPQA/AIME activations of
Qwen3/Phi4) are not available; these seeded draws stand in for them.

Every random stream is derived from ``(seed, tag, index)`` so that one sequence
of a large workload can be regenerated alone (the oracle checks sampled
sequences of full-size workloads that way).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128


def f32(x: float) -> float:
    """A clip ratio as the kernels receive it (an IEEE float32 value)."""
    return float(np.float32(x))


CLIPS_ENVELOPE = tuple(f32(c) for c in (1.00, 0.95, 0.90, 0.85, 0.80))

_TAG_Q, _TAG_K, _TAG_V, _TAG_PROFILE, _TAG_ROT, _TAG_WO, _TAG_TABLE, _TAG_CAL, _TAG_LENS, _TAG_NEW = range(10)


def _rng(seed: int, tag: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(tag), int(index)])


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32.

    Input preparation only: the bf16 workloads are stored as bf16 on the device
    and the oracle reads the same (exactly representable) values.
    """
    x = np.ascontiguousarray(x, dtype=np.float32).copy()
    u = x.view(np.uint32)
    t = (u >> np.uint32(16)) & np.uint32(1)
    t += np.uint32(0x7FFF)
    u += t
    u &= np.uint32(0xFFFF0000)
    return x


def _as_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(f"unsupported input dtype {dtype!r}")


@dataclass
class Rot:
    """A per-KV-head orthogonal rotation, given the way the kernels take it.

    kind: "identity", "signed_hadamard" (R_h = diag(signs_h) H_128 / sqrt(128))
    or "dense" (R_h given as a 128x128 row-major matrix, rows indexed by the
    input channel: x' = x @ R_h).
    """

    kind: str
    signs: np.ndarray | None = None  # [H, 128] float32 of +-1
    dense: np.ndarray | None = None  # [H, 128, 128] float32

    @property
    def n_heads(self) -> int | None:
        if self.signs is not None:
            return self.signs.shape[0]
        if self.dense is not None:
            return self.dense.shape[0]
        return None


def draw_signs(seed: int, index: int, n_heads: int) -> np.ndarray:
    g = _rng(seed, _TAG_ROT, index)
    return np.where(g.random((n_heads, HEAD_DIM)) < 0.5, -1.0, 1.0).astype(np.float32)


def draw_skew_generator(seed: int, index: int, n_heads: int, a_std: float = 0.05) -> np.ndarray:
    """A ~ N(0, a_std^2), one 128x128 matrix per head (float64)."""
    g = _rng(seed, _TAG_ROT, 1000 + index)
    return g.normal(0.0, a_std, size=(n_heads, HEAD_DIM, HEAD_DIM))


def learned_style_rotation(seed: int, index: int, n_heads: int, a_std: float = 0.05) -> np.ndarray:
    """R_h = expm(A_h - A_h^T), the OptR Eq. 11 parameterisation, drawn at random.

    The matrix exponential is SciPy's; the result is an *input* to the kernels
    (a stand-in for a calibrated rotation), stored as float32.
    """
    from scipy.linalg import expm

    a = draw_skew_generator(seed, index, n_heads, a_std)
    out = np.empty((n_heads, HEAD_DIM, HEAD_DIM), dtype=np.float32)
    for h in range(n_heads):
        out[h] = expm(a[h] - a[h].T).astype(np.float32)
    return out


def make_rot(kind: str, seed: int, index: int, n_heads: int, a_std: float = 0.05) -> Rot:
    if kind == "identity":
        return Rot("identity")
    if kind == "signed_hadamard":
        return Rot("signed_hadamard", signs=draw_signs(seed, index, n_heads))
    if kind == "dense":
        return Rot("dense", dense=learned_style_rotation(seed, index, n_heads, a_std))
    raise ValueError(kind)


@dataclass
class KeyProfile:
    """Per-(KV head) outlier channels of the synthetic keys and values."""

    k_channels: np.ndarray  # [H, n_off] int
    k_means: np.ndarray  # [H, n_off] float (+-offset)
    k_std: float
    v_channels: np.ndarray  # [H, n_t] int (Student-t channels)
    v_nu: float


def draw_profile(seed: int, n_kv_heads: int, n_off: int = 6, offset: float = 10.0,
                 k_std: float = 4.0, n_t: int = 2, v_nu: float = 3.0) -> KeyProfile:
    g = _rng(seed, _TAG_PROFILE)
    kc = (np.stack([g.choice(HEAD_DIM, size=n_off, replace=False) for _ in range(n_kv_heads)])
          if n_off else np.zeros((n_kv_heads, 0), int))
    km = np.where(g.random((n_kv_heads, n_off)) < 0.5, -offset, offset)
    vc = (np.stack([g.choice(HEAD_DIM, size=n_t, replace=False) for _ in range(n_kv_heads)])
          if n_t else np.zeros((n_kv_heads, 0), int))
    return KeyProfile(kc, km, k_std, vc, v_nu)


def draw_kv(profile: KeyProfile, seed: int, tag_index: int, n_tok: int, n_kv_heads: int,
            dtype: str) -> tuple[np.ndarray, np.ndarray]:
    """Keys and values [n_tok, H_kv, 128] for one stream (a sequence or a calibration trace)."""
    gk = _rng(seed, _TAG_K, tag_index)
    gv = _rng(seed, _TAG_V, tag_index)
    k = gk.standard_normal((n_tok, n_kv_heads, HEAD_DIM), dtype=np.float32)
    v = gv.standard_normal((n_tok, n_kv_heads, HEAD_DIM), dtype=np.float32)
    for h in range(n_kv_heads):
        for c, m in zip(profile.k_channels[h], profile.k_means[h]):
            k[:, h, c] = (m + profile.k_std * k[:, h, c]).astype(np.float32)
        for c in profile.v_channels[h]:
            v[:, h, c] = gv.standard_t(profile.v_nu, size=n_tok).astype(np.float32)
    return _as_dtype(k, dtype), _as_dtype(v, dtype)


def draw_queries(seed: int, index: int, shape: tuple, dtype: str) -> np.ndarray:
    g = _rng(seed, _TAG_Q, index)
    return _as_dtype(g.standard_normal(shape, dtype=np.float32), dtype)


def draw_wo(seed: int, d_model: int, k_dim: int, dtype: str) -> np.ndarray:
    """W_O [d_model, H_q*128] ~ N(0, 1/k_dim)."""
    g = _rng(seed, _TAG_WO)
    w = g.standard_normal((d_model, k_dim), dtype=np.float32) * np.float32(1.0 / np.sqrt(k_dim))
    return _as_dtype(w, dtype)


def draw_block_table(seed: int, seq_lens, page_tokens: int, num_blocks: int | None = None,
                     shuffle: bool = True) -> tuple[np.ndarray, int]:
    """Block table [n_seqs, max_blocks] (int32, unused entries -1) over a pool
    whose physical pages are handed out in a seeded random order."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    need = (seq_lens + page_tokens - 1) // page_tokens
    total = int(need.sum())
    if num_blocks is None:
        num_blocks = total
    assert num_blocks >= total
    g = _rng(seed, _TAG_TABLE)
    phys = g.permutation(num_blocks)[:total] if shuffle else np.arange(total)
    max_blocks = int(max(1, need.max()))
    table = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = phys[o:o + n]
        o += n
    return table, num_blocks


@dataclass
class DecodeCase:
    """One decode-attention workload: a paged cache of B sequences plus one
    query per query head per sequence."""

    seed: int
    seq_lens: np.ndarray
    n_q_heads: int
    n_kv_heads: int
    d_model: int
    dtype: str
    page_tokens: int
    clip_k: float
    clip_v: float
    rot_k: Rot
    rot_v: Rot
    profile: KeyProfile
    block_table: np.ndarray
    num_blocks: int
    n_cal: int
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_seqs(self) -> int:
        return len(self.seq_lens)

    def kv(self, b: int) -> tuple[np.ndarray, np.ndarray]:
        """Cached keys/values of sequence b: [L_b, H_kv, 128] each."""
        return draw_kv(self.profile, self.seed, b, int(self.seq_lens[b]), self.n_kv_heads, self.dtype)

    def new_kv(self, b: int, n_new: int, step: int = 0) -> tuple[np.ndarray, np.ndarray]:
        """Fresh tokens appended to sequence b (decode-step or prefill-chunk appends)."""
        return draw_kv(self.profile, self.seed, 1_000_000 + 1000 * step + b, n_new, self.n_kv_heads,
                       self.dtype)

    def calibration_keys(self) -> np.ndarray:
        """Keys of a separate calibration trace [n_cal, H_kv, 128] (for the key mean)."""
        k, _ = draw_kv(self.profile, self.seed, 2_000_000, self.n_cal, self.n_kv_heads, self.dtype)
        return k

    def queries(self, step: int = 0) -> np.ndarray:
        return draw_queries(self.seed, step, (self.n_seqs, self.n_q_heads, HEAD_DIM), self.dtype)

    def w_o(self) -> np.ndarray:
        return draw_wo(self.seed, self.d_model, self.n_q_heads * HEAD_DIM, self.dtype)


def decode_case(seed: int, seq_lens, n_q_heads: int, n_kv_heads: int, d_model: int, rot: str,
                dtype: str, page_tokens: int = 16, clip_k: float = 1.0, clip_v: float = 1.0,
                shuffle: bool = True, spare_blocks: int = 0, n_cal: int = 4096,
                n_off: int = 6, name: str = "") -> DecodeCase:
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    need = int(((seq_lens + page_tokens - 1) // page_tokens).sum())
    table, nb = draw_block_table(seed, seq_lens, page_tokens, need + spare_blocks, shuffle)
    return DecodeCase(
        seed=seed, seq_lens=seq_lens, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, d_model=d_model,
        dtype=dtype, page_tokens=page_tokens, clip_k=f32(clip_k), clip_v=f32(clip_v),
        rot_k=make_rot(rot, seed, 0, n_kv_heads), rot_v=make_rot(rot, seed, 1, n_kv_heads),
        profile=draw_profile(seed, n_kv_heads, n_off=n_off), block_table=table, num_blocks=nb,
        n_cal=n_cal, name=name)


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_single_head(seed: int = 1) -> DecodeCase:
    """1 query, 1 KV head, 512 cached fp32 tokens, 4 key channels offset by +8,
    one signed-Hadamard R for K and V, clip 1.0, W_O 128x128 ~ N(0, 1/128)."""
    c = decode_case(seed, [512], 1, 1, 128, "signed_hadamard", "f32", n_off=0, n_cal=512,
                    name="tiny_single_head_512")
    g = _rng(seed, _TAG_PROFILE, 7)
    ch = g.choice(HEAD_DIM, size=4, replace=False)
    c.profile = KeyProfile(ch[None, :], np.full((1, 4), 8.0), 1.0, np.zeros((1, 0), int), 3.0)
    # Same R for K and V, as the workload states.
    c.rot_v = c.rot_k
    return c


def gqa8b_32k(seed: int = 3, n_seqs: int = 16, ctx: int = 32768, page_tokens: int = 16, clip_k: float = 1.0,
              clip_v: float = 1.0) -> DecodeCase:
    """8B-class GQA decode layer: H_q 32, H_kv 8, d_model 4096, bf16, 16 x 32K,
    16-token pages with a shuffled table, dense expm(A - A^T) rotations."""
    return decode_case(seed, [ctx] * n_seqs, 32, 8, 4096, "dense", "bf16", page_tokens=page_tokens,
                       clip_k=clip_k, clip_v=clip_v, name=f"gqa8b_B{n_seqs}_ctx{ctx}")


def long4b_128k(seed: int = 4, n_seqs: int = 1, ctx: int = 131072, page_tokens: int = 16, clip_k: float = 0.9,
                clip_v: float = 0.9) -> DecodeCase:
    """4B-class long-context layer: H_q 32, H_kv 8, d_model 2560, bf16, 128K context,
    signed-Hadamard R per head, clip 0.9 (plus a 4,096-token prefill append)."""
    c = decode_case(seed, [ctx] * n_seqs, 32, 8, 2560, "signed_hadamard", "bf16", page_tokens=page_tokens,
                    clip_k=clip_k, clip_v=clip_v, name=f"long4b_B{n_seqs}_ctx{ctx}")
    c.extra["chunk"] = 4096
    return c


def serve14b_ragged(seed: int = 5, n_seqs: int = 64, page_tokens: int = 16, clip_k: float = 1.0,
                    clip_v: float = 1.0) -> DecodeCase:
    """14B-class serving layer: H_q 40, H_kv 10, d_model 5120, bf16, 64 ragged
    contexts uniform in [1024, 8192], dense per-head R."""
    g = _rng(seed, _TAG_LENS)
    lens = g.integers(1024, 8192 + 1, size=n_seqs)
    return decode_case(seed, lens, 40, 10, 5120, "dense", "bf16", page_tokens=page_tokens, clip_k=clip_k,
                       clip_v=clip_v, n_cal=2560, name=f"serve14b_B{n_seqs}_ragged")


@dataclass
class CalibCase:
    """A candidate-rotation x clip sweep scored by post-W_O NMSE."""

    seed: int
    n_tok: int
    n_qpos: int
    n_kv_heads: int
    gqa: int
    d_model: int
    dtype: str
    k: np.ndarray  # [n_tok, H_kv, 128]
    v: np.ndarray
    q: np.ndarray  # [n_qpos, H_q, 128] -- queries at positions n_tok-n_qpos .. n_tok-1
    w_o: np.ndarray  # [d_model, H_q*128]
    cands: list  # list[Rot], each applied to K and V of every head
    clips: tuple
    joint: bool
    name: str = ""
    fresh_q: np.ndarray | None = None  # evaluation queries [n_fresh, H_q, 128]


def envelope_calibration(seed: int = 6260, n_fresh: int = 10) -> CalibCase:
    """The evaluation page's envelope: 4,096 tokens x 4 KV heads (1 query head
    each), out dim 128, candidates identity + 8 signed-Hadamard, 5 clips, one
    calibration query, then 10 fresh queries."""
    hkv = 4
    prof = draw_profile(seed, hkv)
    k, v = draw_kv(prof, seed, 0, 4096, hkv, "f32")
    q = draw_queries(seed, 0, (1, hkv, HEAD_DIM), "f32")
    fresh = draw_queries(seed, 1, (n_fresh, hkv, HEAD_DIM), "f32")
    w = draw_wo(seed, 128, hkv * HEAD_DIM, "f32")
    cands = [Rot("identity")]
    for i in range(8):
        s = draw_signs(seed, 100 + i, 1)
        cands.append(Rot("signed_hadamard", signs=np.repeat(s, hkv, axis=0)))
    return CalibCase(seed, 4096, 1, hkv, 1, 128, "f32", k, v, q, w, cands, CLIPS_ENVELOPE,
                     joint=True, name="envelope_4096x4", fresh_q=fresh)


def serve14b_calibration(seed: int = 5, n_tok: int = 2560, n_qpos: int = 64, n_cand: int = 16,
                         n_kv_heads: int = 10, gqa: int = 4, d_model: int = 5120) -> CalibCase:
    """Per-head selection over 16 dense candidate rotations x 5 clips on a
    2,560-token calibration trace scored at its final 64 query positions."""
    prof = draw_profile(seed, n_kv_heads)
    k, v = draw_kv(prof, seed, 3_000_000, n_tok, n_kv_heads, "bf16")
    q = draw_queries(seed, 3_000_000, (n_qpos, n_kv_heads * gqa, HEAD_DIM), "bf16")
    w = draw_wo(seed, d_model, n_kv_heads * gqa * HEAD_DIM, "bf16")
    cands = [Rot("dense", dense=learned_style_rotation(seed, 500 + i, n_kv_heads)) for i in range(n_cand)]
    return CalibCase(seed, n_tok, n_qpos, n_kv_heads, gqa, d_model, "bf16", k, v, q, w, cands,
                     CLIPS_ENVELOPE, joint=False, name=f"serve14b_calib_{n_cand}x5")


def small_calibration(seed: int, n_tok: int, n_qpos: int, n_kv_heads: int, gqa: int, d_model: int,
                      kinds=("identity", "signed_hadamard", "dense"), clips=(1.0, 0.9),
                      joint: bool = False, dtype: str = "f32") -> CalibCase:
    prof = draw_profile(seed, n_kv_heads)
    k, v = draw_kv(prof, seed, 0, n_tok, n_kv_heads, dtype)
    q = draw_queries(seed, 0, (n_qpos, n_kv_heads * gqa, HEAD_DIM), dtype)
    w = draw_wo(seed, d_model, n_kv_heads * gqa * HEAD_DIM, dtype)
    cands = [make_rot(kd, seed, 700 + i, n_kv_heads) for i, kd in enumerate(kinds)]
    return CalibCase(seed, n_tok, n_qpos, n_kv_heads, gqa, d_model, dtype, k, v, q, w, cands,
                     tuple(f32(c) for c in clips), joint=joint, name="small_calib")


@dataclass
class OptrHeadCase:
    """One KV head's calibration traces for the OptR gradient calibration: a training
    trace and a held-out trace (queries at the last n_qpos positions, keys, values),
    the head's W_O columns, and base rotations R0_K, R0_V (learned-style, fp64)."""

    seed: int
    gqa: int
    d_model: int
    train: tuple  # (q [n_qpos, gqa, 128], k [n_tok, 128], v [n_tok, 128]) float32
    heldout: tuple
    w_o: np.ndarray  # [d_model, gqa * 128] float32
    r_k0: np.ndarray  # [128, 128] float64
    r_v0: np.ndarray


def optr_head(seed: int, n_tok: int, n_qpos: int, gqa: int, d_model: int, a_std: float = 0.05) -> OptrHeadCase:
    """Synthetic head with the key-outlier profile of the decode workloads (6 offset
    channels), Student-t value channels, N(0,1) queries, W_O ~ N(0, 1/(gqa 128))."""
    prof = draw_profile(seed, 1)
    traces = []
    for i in range(2):
        k, v = draw_kv(prof, seed, 7_000_000 + i, n_tok, 1, "f32")
        q = draw_queries(seed, 7_000_000 + i, (n_qpos, gqa, HEAD_DIM), "f32")
        traces.append((q, k[:, 0, :].copy(), v[:, 0, :].copy()))
    w = draw_wo(seed, d_model, gqa * HEAD_DIM, "f32")
    r_k0 = learned_style_rotation(seed, 900, 1, a_std)[0].astype(np.float64)
    r_v0 = learned_style_rotation(seed, 901, 1, a_std)[0].astype(np.float64)
    return OptrHeadCase(seed, gqa, d_model, traces[0], traces[1], w, r_k0, r_v0)
