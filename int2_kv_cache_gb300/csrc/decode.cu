// Read path: split-K decode attention straight off the packed INT2 pages.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization": Eqs. 1-2 and 5
// (logits <q, k~>/sqrt(d), softmax over the cached positions, o = p^T V~),
// appendix Eqs. 21-22 / 26 (the query is rotated once, q R_K, and meets the
// stored rotated keys), Eq. 27 (the readout stays in the rotated-V basis).
//
// Scale and zero are factored out of the dot products, which is exact algebra:
//   q'.(z + s c)            = s (q'.c) + z sum(q')
//   sum_t p_t (z_t + s_t c_t) = sum_t (p_t s_t) c_t + sum_t p_t z_t
// so both contractions run on the codes c in {0,1,2,3}.
//
// Three kernels per call:
// * qprep_kernel, one CTA per (sequence, KV head): rotates the query heads of
//   the group (Eq. 22), folds in log2(e)/sqrt(128), and lays the result out as
//   the tensor-core B fragments every decode warp loads as is;
// * decode_split_kernel, a fixed grid of 4 CTAs (3 for 8 query heads per KV
//   head) per SM.  The (sequence, KV head, 32-token chunk) list of the whole
//   batch is cut into one contiguous, equal slice per warp, so every warp has
//   the same work whatever the sequence lengths.  A warp streams its chunks
//   through a ring of shared-memory stages (cp.async.bulk copies completed on
//   mbarriers, one page record per lane), and for every (sequence, KV head)
//   unit its slice touches it writes one partial softmax (m, l, unnormalised
//   acc);
// * decode_combine_kernel, one CTA per (unit, query head): the log-sum-exp
//   merge of the unit's partials in a fixed order (deterministic).
// The second and third kernels are programmatic dependent launches: the batch
// scan and the first page copies overlap the query rotation, and the combine
// blocks are scheduled as decode blocks retire.
// With BF16 sink / recent windows (decode_split_kernel<..., true>), positions
// [0, S) and [L - R, L) of a sequence are read from 8-token bf16 records instead
// of the pages: the records form a second list split evenly over the warps,
// staged through the same ring; their keys (centred, not rotated) meet the
// unrotated query, their values (unrotated) are summed apart, and
// decode_combine_win_kernel rotates that sum by R_V once per (unit, query head) (Eq. 27).
// Inside a warp, q'.c and sum_t (p_t s_t) c_t are tensor-core products
// (mma.sync m16n8k16, fp16 inputs, fp32 accumulation).  A 2-bit field masked in
// place inside a 16-bit word is the fp16 value c * 2^(p-24) (a subnormal, p =
// the field's bit offset), so the operands need one logical operation per two
// codes, and the power-of-two factor is compensated exactly in the other
// operand.  The value codes are read transposed (ldmatrix .trans) so that each
// register holds two tokens of one channel group, as the product wants.  The
// fp32 operand of each product (the rotated query, the weights p_t s_t) is
// split into an fp16 high part and an fp16 remainder occupying the two MMA
// columns of one head, which keeps ~22 significant bits.  The softmax runs
// online in base 2 with a lazy reference maximum.
#include <type_traits>

#include "async_copy.cuh"
#include "quant_common.cuh"

namespace kvq {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int DEC_WARPS = 4;   // warps (slices) per work partition
constexpr int DEC_STAGES = 3;  // stages of 64 tokens per warp
// Lazy softmax rescaling: the running sums keep their reference maximum until a
// chunk's maximum exceeds it by more than TAU (log2 units), so weights stay <= 2^TAU.
constexpr float TAU = 6.f;
// The fp16 remainder column carries (x - fp16(x)) * 2^11, keeping it out of the
// subnormal range whenever the high part is normal.
constexpr float LO_SCALE = 2048.f;
constexpr float LO_UNSCALE = 1.f / 2048.f;
constexpr int PART = D + 4;  // floats per head in a partial: acc[128], m (log2 units), l, 2 pad (16-byte rows)

// Work partitions of 4 warps resident per SM (register bound: 128 or 170 per thread).
__host__ __device__ constexpr int ctas_per_sm(int gqa) { return gqa >= 8 ? 3 : 4; }
// Largest thread block of the decode kernel: every partition of one SM in one block.
__host__ __device__ constexpr int dec_max_warps(int gqa) { return DEC_WARPS * ctas_per_sm(gqa); }
__host__ __device__ constexpr int n_tiles(int gqa) { return (gqa + 3) / 4; }

// Workspace regions (each 256-byte aligned):
//   part   [n_slots][gqa][132] fp32 partials, n_slots = 4 * n_ctas + U; the
//          partial of warp w for unit u lives in slot w + u (the units a warp
//          slice touches are consecutive, so slots never collide)
//   qfrag  [U][16 * NT][32] u32: query B fragments, lane-major
//   qconst [U][gqa][4] fp32: dscale, sum(q')/dscale, TAU/dscale, 0
//   span   [U] int2: the warp slices (k0, k1) that meet the unit, (1, 0) if none
// and, with BF16 windows, the same for the window-record list:
//   partw  [n_slots][gqa][132] fp32, wqfrag [U][16 * NT][32] u32 (bf16 pairs), spanw [U] int2
// with U = n_seqs * n_kv_heads units (sequence b, KV head h) -> u = b * n_kv_heads + h.
struct DecWs {
  float* part;
  uint32_t* qfrag;
  float* qconst;
  int2* span;
  float* partw;       // nullptr without windows
  uint32_t* wqfrag;
  int2* spanw;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t decode_ws_layout(void* base, int n_seqs, int n_kv_heads, int gqa, int n_ctas,
                                                   bool windows, DecWs* out) {
  const size_t units = (size_t)n_seqs * n_kv_heads;
  const size_t slots = (size_t)DEC_WARPS * n_ctas + units;
  const size_t frag_bytes = units * 16 * n_tiles(gqa) * 32 * sizeof(uint32_t);
  const size_t o_part = 0;
  const size_t o_frag = align256(o_part + slots * gqa * PART * sizeof(float));
  const size_t o_const = align256(o_frag + frag_bytes);
  const size_t o_span = align256(o_const + units * gqa * 4 * sizeof(float));
  const size_t o_partw = align256(o_span + units * sizeof(int2));
  size_t total = o_partw;
  size_t o_wfrag = 0, o_spanw = 0;
  if (windows) {
    o_wfrag = align256(o_partw + slots * gqa * PART * sizeof(float));
    o_spanw = align256(o_wfrag + frag_bytes);
    total = align256(o_spanw + units * sizeof(int2));
  }
  if (out) {
    char* p = static_cast<char*>(base);
    out->part = reinterpret_cast<float*>(p + o_part);
    out->qfrag = reinterpret_cast<uint32_t*>(p + o_frag);
    out->qconst = reinterpret_cast<float*>(p + o_const);
    out->span = reinterpret_cast<int2*>(p + o_span);
    out->partw = windows ? reinterpret_cast<float*>(p + o_partw) : nullptr;
    out->wqfrag = windows ? reinterpret_cast<uint32_t*>(p + o_wfrag) : nullptr;
    out->spanw = windows ? reinterpret_cast<int2*>(p + o_spanw) : nullptr;
  }
  return total;
}

size_t decode_workspace_bytes(int n_seqs, int n_kv_heads, int gqa, int n_ctas, bool windows) {
  return decode_ws_layout(nullptr, n_seqs, n_kv_heads, gqa, n_ctas, windows, nullptr);
}

// Default grid: a full single wave (4 or 3 CTAs per SM), but no more warps than
// slices of at least four chunks.
int decode_auto_ctas(int n_seqs, int n_kv_heads, int gqa, int max_seq_len) {
  const long long chunks = (long long)n_seqs * n_kv_heads * ((max_seq_len + 31) / 32);
  const long long by_work = (chunks + 4 * DEC_WARPS - 1) / (4 * DEC_WARPS);
  long long n = (long long)device_sm_count() * ctas_per_sm(gqa);
  if (n > by_work) n = by_work;
  return n < 1 ? 1 : (int)n;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The same product with a zero accumulator input (d = A B).
__device__ __forceinline__ void mma16816_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
// bf16 operands (the BF16 window records)
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma16816_bf16_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                   uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float half_rn(float x) { return __half2float(__float2half_rn(x)); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A chunk = two 16-token tiles of one sequence and KV head, staged as 2 page
// records (16-token pages) or 4 (8-token pages).  Byte offsets of row r (0..15)
// of tile u (0, 1) inside the staged chunk:
template <int P>
struct ChunkLayout {
  static __device__ __forceinline__ int base(int u, int r) {
    return P == 16 ? u * 1152 : (2 * u + (r >> 3)) * 576;
  }
  static __device__ __forceinline__ int rr(int r) { return P == 16 ? r : (r & 7); }
  static __device__ __forceinline__ int k(int u, int r) { return base(u, r) + 32 * rr(r); }
  static __device__ __forceinline__ int v(int u, int r) { return base(u, r) + 32 * P + 32 * rr(r); }
  static __device__ __forceinline__ int km(int u, int r) { return base(u, r) + 64 * P + 4 * rr(r); }
  static __device__ __forceinline__ int vm(int u, int r) { return base(u, r) + 68 * P + 4 * rr(r); }
  static __device__ __forceinline__ int page(int u, int r) { return P == 16 ? u : 2 * u + (r >> 3); }
};

// (scale, zero) fp16 pair of one token -> fp32
__device__ __forceinline__ float2 meta_pair(const uint8_t* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}

// Value codes are read with a transposing shared-memory load (ldmatrix .trans):
// each register then holds one 16-bit element (8 channels) of two consecutive
// tokens.  Field f (channel 8e + f) is masked in place for f = 1..4 (bit 2f)
// and from the byte-swapped word for f = 0, 5, 6, 7 (bits 8, 2, 4, 6), so its
// fp16 value is c * 2^(pe-24) with pe in {2, 4, 6, 8}.
__host__ __device__ constexpr int v_pe(int f) { return f == 0 ? 8 : (f <= 4 ? 2 * f : 2 * f - 8); }
__host__ __device__ constexpr bool v_swapped(int f) { return f == 0 || f >= 5; }


// ---------------------------------------------------------------------------
// The new token of a decode step (kvq_decode_step): its key and value groups
// are quantized and written by the query-preparation CTA of (sequence, KV head),
// with the decisions of the cache-write kernels (OptR §6 cache-write kernel;
// Eqs. 4, 20, 21, 27):
//   x = k R_K - mu R_K (keys) or v R_V (values); lo = c min x, hi = c max x;
//   scale = fp16((hi - lo)/3), zero = fp16(lo), code = clamp(rint((x - zero)/scale), 0, 3).
// Dense R: warp w forms the partial x R over rows 16w .. 16w + 15 of R_h in
// double-float (error-free products and sums; app_df_partial) and one warp adds
// the 8 partials in a fixed tree and decides exactly (app_df_decide).  A step
// appends one token per (sequence, head), so the exact path costs little and
// takes no uncertain second pass (the query preparation gates the whole decode,
// so its slowest CTA counts).  The key meets the rows of R_K that the query
// rotation holds in registers; R_V is staged in shared memory by bulk copies
// issued when the CTA starts.  Identity / signed Hadamard: one warp, certified
// fp32 or a double-float redo (app_warp).
// ---------------------------------------------------------------------------
struct AppSmem {     // per role (key, value)
  float2 df[8][D];   // each warp's partial x R as (hi, lo)
  float x[D];        // the input row
};

__device__ __forceinline__ void app_write(uint8_t* codes, uint8_t* meta, unsigned byte, const QParams& qp, int lane) {
  codes[lane] = (uint8_t)byte;
  if (lane == 0) *reinterpret_cast<uint32_t*>(meta) = (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
}

// Every warp: its 16 rows' partial x R in double-float.
__device__ __forceinline__ void app_df_partial(const float* __restrict__ s_x, const float4 (&rr)[16], int warp,
                                               int lane, AppSmem& a) {
  float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float xc = s_x[16 * warp + r];
    const float rv[4] = {rr[r].x, rr[r].y, rr[r].z, rr[r].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __fmul_rn(xc, rv[i]);
      const float pe = __fmaf_rn(xc, rv[i], -p);
      const DF t = two_sum(sh[i], p);
      sh[i] = t.hi;
      sl[i] = __fadd_rn(sl[i], __fadd_rn(t.lo, pe));
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const DF c = df_norm(sh[i], sl[i]);
    a.df[warp][4 * lane + i] = make_float2(c.hi, c.lo);
  }
}

// One warp: adds the double-float partials in a fixed tree, subtracts mu R (if given)
// and decides exactly.
__device__ __forceinline__ void app_df_decide(const AppSmem& a, bool has_mu, float4 mu, float clip, uint8_t* codes,
                                              uint8_t* meta, int lane) {
  DF x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    DF q[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) q[w] = DF{a.df[w][4 * lane + i].x, a.df[w][4 * lane + i].y};
    x[i] = df_add(df_add(df_add(q[0], q[1]), df_add(q[2], q[3])), df_add(df_add(q[4], q[5]), df_add(q[6], q[7])));
  }
  if (has_mu) {
    x[0] = df_add_f(x[0], -mu.x); x[1] = df_add_f(x[1], -mu.y);
    x[2] = df_add_f(x[2], -mu.z); x[3] = df_add_f(x[3], -mu.w);
  }
  QParams qp;
  const unsigned byte = quantize_warp_df(x, clip, qp);
  app_write(codes, meta, byte, qp, lane);
}

// One warp, identity or signed Hadamard: certified fp32, else double-float.
__device__ __forceinline__ void app_warp(const float* __restrict__ s_x, const RotDev& rot, int h,
                                         const float* __restrict__ mu_rot, float clip, uint8_t* codes, uint8_t* meta,
                                         int lane) {
  const float4 v = reinterpret_cast<const float4*>(s_x)[lane];
  float4 mu = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mu_rot) mu = __ldg(reinterpret_cast<const float4*>(mu_rot + (size_t)h * D) + lane);
  float y[4] = {v.x, v.y, v.z, v.w};
  float E = rotate_f32_bounded(y, rot, h, lane);
  if (mu_rot) {
    y[0] = __fsub_rn(y[0], mu.x); y[1] = __fsub_rn(y[1], mu.y);
    y[2] = __fsub_rn(y[2], mu.z); y[3] = __fsub_rn(y[3], mu.w);
    // the subtraction's rounding: u (|y| + |mu|), y bounded through E's l1 norm or |x|
    E += (warp_max(fmaxf(fmaxf(fabsf(v.x) + fabsf(mu.x), fabsf(v.y) + fabsf(mu.y)),
                         fmaxf(fabsf(v.z) + fabsf(mu.z), fabsf(v.w) + fabsf(mu.w)))) +
          E * 524288.f) * P2_M22;
  }
  QParams qp;
  unsigned byte = 0u;
  if (!quantize_warp_certain(y, E, clip, qp, byte)) {
    DF x[4] = {{v.x, 0.f}, {v.y, 0.f}, {v.z, 0.f}, {v.w, 0.f}};
    rotate_df_warp(x, rot, h, lane);
    if (mu_rot) {
      x[0] = df_add_f(x[0], -mu.x); x[1] = df_add_f(x[1], -mu.y);
      x[2] = df_add_f(x[2], -mu.z); x[3] = df_add_f(x[3], -mu.w);
    }
    byte = quantize_warp_df(x, clip, qp);
  }
  app_write(codes, meta, byte, qp, lane);
}

// Dynamic shared memory of the query preparation with a step's append: R_V staged
// (dense values only), then the two roles' AppSmem.
constexpr int QPA_RV_BYTES = D * D * 4;
__host__ __device__ constexpr int qpa_smem_bytes(bool dense_v) {
  return (dense_v ? QPA_RV_BYTES : 0) + 2 * (int)sizeof(AppSmem);
}

// ---------------------------------------------------------------------------
// Query preparation (Eq. 22), one CTA per (KV head h, sequence b), 256 threads
// (with a decode step's append it also writes the new token's key and value,
// see above):
// q'_j = q[b][h G + j] R_K,h * log2(e)/sqrt(128) for the G query heads of the
// group, then per head the sum of q' and a power-of-two prescale e_j keeping
// 256 |q'| well inside the fp16 range, and the B fragments of q'.c.  Also
// marks the unit as not yet covered and writes o = 0 for an empty sequence.
// ---------------------------------------------------------------------------
constexpr int QP_THREADS = 256;

template <int G, bool DENSE, bool APPEND, bool WAPP = false>  // WAPP: the append also writes a window row
__global__ void __launch_bounds__(QP_THREADS) qprep_kernel(int n_q_heads, int n_kv_heads, const void* __restrict__ q,
                                                           int q_dtype, RotDev rot, const int32_t* __restrict__ seq_lens,
                                                           DecWs ws, float* __restrict__ o_rot, PageGeom pg,
                                                           const int32_t* __restrict__ table, StepAppend app,
                                                           unsigned* err, int n_seqs, int seqs_per_cta) {
  constexpr int NT = n_tiles(G);
  constexpr int NW = QP_THREADS / 32;
  pdl_launch_dependents();  // the decode kernel may start its batch scan and first copies
  __shared__ __align__(16) float qv[G][D];
  __shared__ __align__(16) float qr[G][D];
  __shared__ __align__(16) float red[DENSE ? NW : 1][G][D];
  __shared__ float qe[G];
  const int h = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float sc = LOG2E * INV_SQRT_D;
  // ---- a decode step's new token (APPEND): where it goes, its rows, R_V in flight ----
  extern __shared__ __align__(128) uint8_t qpa_dyn[];  // APPEND: [R_V (dense values)][AppSmem key][AppSmem value]
  __shared__ __align__(8) uint64_t rv_bar;
  const bool dense_v = APPEND && app.rot_v.kind == KVQ_ROT_DENSE;
  const float4* sRV = reinterpret_cast<const float4*>(qpa_dyn);
  AppSmem* ak = reinterpret_cast<AppSmem*>(qpa_dyn + (dense_v ? QPA_RV_BYTES : 0));
  AppSmem* av = ak + 1;
  int new_len = 0;  // the deciding warps (NW - 1: key, NW - 2: value): seq_lens[b], loaded early
  float4 mu_k = make_float4(0.f, 0.f, 0.f, 0.f);  // warp NW - 1: its channels of mu R_K
  if (APPEND && tid == 0 && dense_v) {
      mbar_init(&rv_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&rv_bar, QPA_RV_BYTES);
      fence_proxy_async();
      const uint8_t* src = reinterpret_cast<const uint8_t*>(app.rot_v.dense + (size_t)h * D * D);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        bulk_g2s(qpa_dyn + c * (QPA_RV_BYTES / 4), src + c * (QPA_RV_BYTES / 4), QPA_RV_BYTES / 4, &rv_bar);
  }
  if (APPEND && warp == NW - 1 && app.mu_rot_k)
    mu_k = __ldg(reinterpret_cast<const float4*>(app.mu_rot_k + (size_t)h * D) + lane);
  // warp w: rows 16w .. 16w + 15 of R_K, lane: columns 4l .. 4l + 3, loaded once for the
  // CTA's sequences (all row loads in flight at once)
  float4 r[16];
  if (DENSE) {
    const float4* R = reinterpret_cast<const float4*>(rot.dense + (size_t)h * D * D) + lane;
#pragma unroll
    for (int c = 0; c < 16; ++c) r[c] = __ldg(R + (size_t)(16 * warp + c) * (D / 4));
  }
  // ---- the CTA's sequences: blockIdx.y * seqs_per_cta + si ----
  for (int si = 0; si < seqs_per_cta; ++si) {
  const int b = blockIdx.y * seqs_per_cta + si;
  if (b >= n_seqs) break;
  const int u = b * n_kv_heads + h;
  if (si > 0) __syncthreads();  // the previous sequence's readers of the shared buffers are done
  if (APPEND) {
    const size_t e0 = ((size_t)b * n_kv_heads + h) * D;
    if (warp == NW - 1) {
      new_len = __ldg(seq_lens + b);
      reinterpret_cast<float4*>(ak->x)[lane] = load4(app.k, e0 + 4 * lane, app.dtype);
    }
    if (warp == NW - 2) {
      new_len = __ldg(seq_lens + b);
      reinterpret_cast<float4*>(av->x)[lane] = load4(app.v, e0 + 4 * lane, app.dtype);
    }
    if (!DENSE) __syncthreads();  // the dense path's first barrier covers these writes
  }
  // The new token's page record (position len - 1; none for an empty sequence, nothing for
  // a position or block id out of range, which the key's warp flags), by the deciding warps.
  auto new_record = [&](int& slot) -> uint8_t* {
    const int len = new_len;
    if (len < 1 || len > pg.max_blocks * pg.page_tokens) return nullptr;
    const int pos = len - 1;
    const int blk = __ldg(table + (size_t)b * pg.max_blocks + pos / pg.page_tokens);
    if (blk < 0 || blk >= pg.num_blocks) {
      if (warp == NW - 1 && lane == 0) flag_error(err, ERR_BLOCK_RANGE);
      return nullptr;
    }
    slot = pos % pg.page_tokens;
    return app.pool + ((size_t)blk * n_kv_heads + h) * pg.record;
  };
  if (DENSE) {
    for (int i = tid; i < G * D; i += QP_THREADS)
      qv[i / D][i % D] = load1(q, ((size_t)b * n_q_heads + h * G) * D + i, q_dtype);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float x = qv[j][16 * warp + c];
        a.x = fmaf(x, r[c].x, a.x); a.y = fmaf(x, r[c].y, a.y); a.z = fmaf(x, r[c].z, a.z); a.w = fmaf(x, r[c].w, a.w);
      }
      reinterpret_cast<float4*>(red[warp][j])[lane] = a;
    }
    if (APPEND) app_df_partial(ak->x, r, warp, lane, *ak);  // the new key meets the same rows of R_K
    __syncthreads();
    for (int i = tid; i < G * D; i += QP_THREADS) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) a += red[w][i / D][i % D];
      qr[i / D][i % D] = a * sc;
    }
  } else {
    for (int j = warp; j < G; j += NW) {
      float4 x = load4(q, ((size_t)b * n_q_heads + h * G + j) * D + 4 * lane, q_dtype);
      x = rotate_vec_warp(x, rot, h, lane, false);
      x.x *= sc; x.y *= sc; x.z *= sc; x.w *= sc;
      reinterpret_cast<float4*>(qr[j])[lane] = x;
    }
  }
  if (APPEND) {
    // values with a dense R_V: every warp its 16 staged rows, in double-float
    if (dense_v) {
      if (!mbar_wait_bounded(&rv_bar, 0)) {
        if (tid == 0) flag_error(err, ERR_TIMEOUT);
      } else {
        float4 rv[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) rv[c] = sRV[(16 * warp + c) * 32 + lane];
        app_df_partial(av->x, rv, warp, lane, *av);
      }
    }
    __syncthreads();
    // with BF16 windows, warp 0 writes the new token's window row (the rules of
    // window_append_kernel: key = bf16(k - mu), value = bf16(v); sink slot p < S, else
    // recent slot S + p % R)
    if (WAPP && warp == 0) {
      const int len = __ldg(seq_lens + b), p = len - 1;
      const int S = app.win.sink, R = app.win.recent;
      if (len >= 1 && len <= pg.max_blocks * pg.page_tokens && (p < S || R > 0)) {
        const int slot = p < S ? p : S + p % R;
        uint8_t* wrec = app.win.buf + (((size_t)b * n_kv_heads + h) * ((S + R) / WIN_REC_TOKENS) +
                                       slot / WIN_REC_TOKENS) * WIN_REC_BYTES;
        const int row = slot % WIN_REC_TOKENS;
        const int off = row * 256 + (((lane >> 1) ^ row) << 4) + (lane & 1) * 8;
        float4 x = reinterpret_cast<const float4*>(ak->x)[lane];
        if (app.mu_win) {
          const float4 m = __ldg(reinterpret_cast<const float4*>(app.mu_win + (size_t)h * D) + lane);
          x = make_float4(__fsub_rn(x.x, m.x), __fsub_rn(x.y, m.y), __fsub_rn(x.z, m.z), __fsub_rn(x.w, m.w));
        }
        const float4 y = reinterpret_cast<const float4*>(av->x)[lane];
        const __nv_bfloat162 k01 = __floats2bfloat162_rn(x.x, x.y), k23 = __floats2bfloat162_rn(x.z, x.w);
        const __nv_bfloat162 v01 = __floats2bfloat162_rn(y.x, y.y), v23 = __floats2bfloat162_rn(y.z, y.w);
        *reinterpret_cast<uint2*>(wrec + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&k01), *reinterpret_cast<const uint32_t*>(&k23));
        *reinterpret_cast<uint2*>(wrec + 2048 + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&v01), *reinterpret_cast<const uint32_t*>(&v23));
      }
    }
    // the decisions: warp NW - 1 the key, warp NW - 2 the value (dense: the exact
    // decision on the double-float partials; otherwise the one-warp path)
    const int P = pg.page_tokens;
    if (warp == NW - 1) {
      int slot = 0;
      uint8_t* rec = new_record(slot);
      if (rec) {
        if (DENSE) app_df_decide(*ak, app.mu_rot_k != nullptr, mu_k, app.clip_k, rec + 32 * slot, rec + 64 * P + 4 * slot, lane);
        else app_warp(ak->x, rot, h, app.mu_rot_k, app.clip_k, rec + 32 * slot, rec + 64 * P + 4 * slot, lane);
      }
    }
    if (warp == NW - 2) {
      int slot = 0;
      uint8_t* rec = new_record(slot);
      if (rec) {
        if (dense_v)
          app_df_decide(*av, false, mu_k, app.clip_v, rec + 32 * P + 32 * slot, rec + 68 * P + 4 * slot, lane);
        else
          app_warp(av->x, app.rot_v, h, nullptr, app.clip_v, rec + 32 * P + 32 * slot, rec + 68 * P + 4 * slot, lane);
      }
    }
    // the decode kernel reads the pages with bulk copies (the async proxy)
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  __syncthreads();
  for (int j = warp; j < G; j += NW) {
    const float4 v = reinterpret_cast<const float4*>(qr[j])[lane];
    const float tot = warp_sum(v.x + v.y + v.z + v.w);
    const float mx = warp_max(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    if (lane == 0) {
      int e = 0;
      while (e < 64 && mx * 256.f > 16384.f * exp2f((float)e)) ++e;
      qe[j] = (float)e;
      const float inv = exp2f(-16.f - (float)e);
      reinterpret_cast<float4*>(ws.qconst)[(size_t)u * G + j] = make_float4(exp2f(16.f + (float)e), tot * inv, TAU * inv, 0.f);
    }
  }
  __syncthreads();
  // B fragment word (nt, s, r) of lane (g, t): column g <-> head j = 4nt + g/2,
  // the fp16 high part (g even) or the remainder * 2^11 (g odd) of
  // q'_j * 2^(8 - pe - e_j) at channels 32t + 16r + s and 32t + 16r + 8 + s, the
  // key field of k-slice s sitting at bit pe = 2s (s <= 4) or 2s - 10.
  uint32_t* fr = ws.qfrag + (size_t)u * NT * 16 * 32;
  for (int wv = tid; wv < NT * 16 * 32; wv += QP_THREADS) {
    const int w = wv >> 5, L = wv & 31;
    const int nt = w >> 4, s = (w & 15) >> 1, r = w & 1;
    const int gi = L >> 2, ti = L & 3;
    const int j = 4 * nt + (gi >> 1);
    const int pe = s <= 4 ? 2 * s : 2 * s - 10;
    float v0 = 0.f, v1 = 0.f;
    if (j < G) {
      const float f = exp2f((float)(8 - pe) - qe[j]);
      const float x0 = qr[j][32 * ti + 16 * r + s] * f, x1 = qr[j][32 * ti + 16 * r + 8 + s] * f;
      const float h0 = half_rn(x0), h1 = half_rn(x1);
      v0 = (gi & 1) ? (x0 - h0) * LO_SCALE : h0;
      v1 = (gi & 1) ? (x1 - h1) * LO_SCALE : h1;
    }
    fr[wv] = pack_half2(v0, v1);
  }
  if (ws.wqfrag) {
    // window B fragments: the UNROTATED q_j * log2(e)/sqrt(128) (window keys are
    // not rotated, Eq. 24), as bf16 high part (column g even) and bf16 remainder
    // (g odd) at channels 16 s + 2t + 8 r and 16 s + 2t + 8 r + 1
    uint32_t* wf = ws.wqfrag + (size_t)u * NT * 16 * 32;
    for (int wv = tid; wv < NT * 16 * 32; wv += QP_THREADS) {
      const int w = wv >> 5, L = wv & 31;
      const int nt = w >> 4, s = (w & 15) >> 1, r = w & 1;
      const int gi = L >> 2, ti = L & 3;
      const int j = 4 * nt + (gi >> 1);
      uint32_t word = 0u;
      if (j < G) {
        const size_t e0 = ((size_t)b * n_q_heads + h * G + j) * D + 16 * s + 2 * ti + 8 * r;
        const float x0 = load1(q, e0, q_dtype) * sc, x1 = load1(q, e0 + 1, q_dtype) * sc;
        __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
        if (gi & 1) {
          h0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
          h1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
        }
        word = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      }
      wf[wv] = word;
    }
    if (tid == 0) ws.spanw[u] = make_int2(1, 0);
  }
  if (tid == 0) ws.span[u] = make_int2(1, 0);
  if (__ldg(seq_lens + b) == 0)  // no cached tokens: the softmax is over nothing, o = 0
    for (int i = tid; i < G * D; i += QP_THREADS) o_rot[((size_t)b * n_q_heads + h * G) * D + i] = 0.f;
  }
}

// Position of a warp in the batch's chunk list: unit (sequence b, KV head h)
// covering list entries [S, E), nb = chunks of b, len = cached tokens of b.
struct ChunkWalker {
  int b, h, len, nb, S, E;
};

// ---------------------------------------------------------------------------
// The decode kernel.  Each warp works through its own slice of the chunk list;
// the warps are grouped into blocks of nw = blockDim.x / 32 (4 .. dec_max_warps)
// and only the total number of warps decides the slices (and so the result).
// A full wave runs as one block per SM: the warps of one block progress at the
// same rate, while several blocks on one SM finish one after another in the
// order they arrived, which leaves the SM partly idle at the end.
// G = query heads per KV head; NT = n-tiles of 8 columns (2 columns per head).
// ---------------------------------------------------------------------------
template <int G, int P, bool WIN>
__global__ void __launch_bounds__(dec_max_warps(G) * 32, 1) decode_split_kernel(
    PageGeom g, int n_seqs, int n_q_heads, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ table, const uint8_t* __restrict__ pool, DecWs ws,
    float* __restrict__ o_rot, unsigned* err, WinGeom win, int step_append) {
  constexpr int NT = n_tiles(G);
  constexpr int NST = DEC_STAGES;
  constexpr int PPC = 32 / P;              // pages per 32-token chunk
  constexpr int REC = 72 * P;              // bytes per page record
  constexpr int CHUNK = PPC * REC;         // 2304 bytes: one 32-token chunk
  constexpr int PPS = 2 * PPC;             // pages per stage (64 tokens)
  constexpr int STAGE = 2 * CHUNK;         // 4608 bytes
  constexpr int CPF = 32 / PPS;            // stages per fill of the page cache
  constexpr uint32_t ALL_PAGES = (1u << PPS) - 1u;
  constexpr uint32_t CHUNK_PAGES = (1u << PPC) - 1u;
  constexpr unsigned FULLM = 0xffffffffu;
  using CL = ChunkLayout<P>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;  // MMA group id, thread id in group
  const int Hkv = g.n_kv_heads;
  const int max_len = g.max_blocks * P;
  // BF16 windows: positions [0, S_w) and [len - R_w, len) are read from the window records
  const int S_w = WIN ? win.sink : 0, R_w = WIN ? win.recent : 0;
  const int n_wrec = (S_w + R_w) / WIN_REC_TOKENS;  // records per (sequence, KV head)

  constexpr int MAXW = dec_max_warps(G);
  const int nw = blockDim.x >> 5;  // warps of this block
  extern __shared__ __align__(128) uint8_t dyn_smem[];  // [nw][DEC_STAGES][STAGE]
  auto stage_ptr = [&](int w, int sidx) { return dyn_smem + (w * DEC_STAGES + sidx) * STAGE; };
  __shared__ __align__(8) uint64_t bars[MAXW][DEC_STAGES];
  __shared__ uint8_t sflag[MAXW][DEC_STAGES];  // bit p: page p of the staged entry was copied
  __shared__ int s_sum[MAXW], s_sumw[MAXW];
  __shared__ int s_start[MAXW][3];   // first sequence of each warp's slice, entries before it, its length
  __shared__ int s_startw[MAXW][3];  // the same for the window-record list

  // list entries (64-token stages) of a sequence of `len` tokens: INT2 positions [S_w, len - R_w)
  auto n_chunks_of = [&](int len) {
    if (len <= 0 || len > max_len) return 0;
    const int e = len - R_w;
    return e > S_w ? (e - S_w + 63) >> 6 : 0;
  };
  // window records of a sequence of `len` tokens: the sink [0, min(S_w, len)) in records
  // of 8 positions, then the recent part [max(S_w, len - R_w), len) by 8-aligned groups
  auto n_wrec_of = [&](int len) {
    if (!WIN || len <= 0 || len > max_len) return 0;
    const int a = max(S_w, len - R_w);
    return ((min(S_w, len) + 7) >> 3) + (a < len ? ((len + 7) >> 3) - (a >> 3) : 0);
  };

  // ---- the batch's chunk list: sequence b holds H_kv * nb_b entries, unit (b, h)
  //      the nb_b entries from H_kv * prefix_b + h * nb_b on ----
  // the lengths are kept in the (still unused) stage memory for the second pass
  int* s_len = reinterpret_cast<int*>(dyn_smem);
  const bool cached = n_seqs <= nw * DEC_STAGES * STAGE / (int)sizeof(int);
  auto len_of = [&](int b) { return cached ? s_len[b] : __ldg(seq_lens + b); };
  int tot = 0, totw = 0;
  for (int b = threadIdx.x; b < n_seqs; b += blockDim.x) {
    const int len = __ldg(seq_lens + b);
    if ((len < 0 || len > max_len) && blockIdx.x == 0) flag_error(err, ERR_SEQ_RANGE);
    if (cached) s_len[b] = len;
    tot += n_chunks_of(len);
    if (WIN) totw += n_wrec_of(len);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(FULLM, tot, o);
    if (WIN) totw += __shfl_xor_sync(FULLM, totw, o);
  }
  if (lane == 0) {
    s_sum[warp] = tot;
    s_sumw[warp] = totw;
  }
  __syncthreads();
  int T = 0, Tws = 0;
  for (int w = 0; w < nw; ++w) {
    T += s_sum[w];
    Tws += s_sumw[w];
  }
  T *= Hkv;
  const int n_warps = gridDim.x * nw;
  const int Ww = (T + n_warps - 1) / n_warps;  // entries per warp slice
  const int gw = blockIdx.x * nw + warp;
  const int ga = min(T, gw * Ww);
  const int my_n = min(T, ga + Ww) - ga;
  // the window records are split the same way, in a list of their own
  const int Tw = WIN ? Hkv * Tws : 0;
  const int Wwn = (Tw + n_warps - 1) / n_warps;
  const int gaw = min(Tw, gw * Wwn);
  const int my_nw = min(Tw, gaw + Wwn) - gaw;
  const int F = my_n + my_nw;  // stage fills of this warp
  __syncthreads();
  // exclusive prefix of per-sequence counts, tile by tile: the sequence holding
  // the first entry of each warp slice of a list (W entries per slice, Ttot in all)
  auto find_starts = [&](auto count, int W, int Ttot, int (*st)[3]) {
    int base = 0;
    for (int b0 = 0; b0 < n_seqs; b0 += blockDim.x) {
      const int b = b0 + threadIdx.x;
      const int len = b < n_seqs ? len_of(b) : 0;
      const int n = count(len);
      int inc = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULLM, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) s_sum[warp] = inc;
      __syncthreads();
      int before = base;
      for (int w = 0; w < warp; ++w) before += s_sum[w];
      const int excl = before + inc - n;
      if (n > 0) {
        for (int w = 0; w < nw; ++w) {
          const int gs = (blockIdx.x * nw + w) * W;
          if (gs < Ttot && gs >= Hkv * excl && gs < Hkv * (excl + n)) {
            st[w][0] = b;
            st[w][1] = excl;
            st[w][2] = len;
          }
        }
      }
      for (int w = 0; w < nw; ++w) base += s_sum[w];
      __syncthreads();
    }
  };
  find_starts(n_chunks_of, Ww, T, s_start);
  if (WIN) find_starts(n_wrec_of, Wwn, Tw, s_startw);
  // advance a walker to list entry gq (entries per sequence from `count`)
  auto walk_gen = [&](ChunkWalker& w, int gq, auto count) {
    while (gq >= w.E) {
      if (++w.h == Hkv) {
        w.h = 0;
        ++w.b;
        w.len = __ldg(seq_lens + w.b);
        w.nb = count(w.len);
      }
      w.S = w.E;
      w.E = w.S + w.nb;
    }
  };
  auto walk_to = [&](ChunkWalker& w, int gq) { walk_gen(w, gq, n_chunks_of); };
  auto walk_w = [&](ChunkWalker& w, int gq) { walk_gen(w, gq, n_wrec_of); };
  auto init_walker = [&](ChunkWalker& w, const int* st, int g0, auto count) {
    w.b = st[0];
    w.len = st[2];
    w.nb = count(w.len);
    const int sb = Hkv * st[1];
    w.h = (g0 - sb) / w.nb;
    w.S = sb + w.h * w.nb;
    w.E = w.S + w.nb;
  };
  ChunkWalker iw, iww;  // issue side: INT2 list, window list
  if (my_n > 0) init_walker(iw, s_start[warp], ga, n_chunks_of);
  if (WIN && my_nw > 0) init_walker(iww, s_startw[warp], gaw, n_wrec_of);
  ChunkWalker cw = iw, cww = iww;  // consume side

  // Page cache: lane l holds the record index (block * H_kv + h) of page l % PPS
  // of the warp's entry i0 + l / PPS; -2: past the sequence, -1: bad block id.
  int rec = -2;
  int n_issued = 0;  // chunks whose copies were issued
  auto fill_cache = [&](int i0) {
    ChunkWalker w = iw;
    const int i = i0 + lane / PPS;
    rec = -2;
    if (i < my_n) {
      walk_to(w, ga + i);
      const int pg = S_w / P + (ga + i - w.S) * PPS + lane % PPS;
      if (pg < (w.len - R_w + P - 1) / P) {
        const int pid = __ldg(table + (size_t)w.b * g.max_blocks + pg);
        rec = (pid >= 0 && pid < g.num_blocks) ? pid * Hkv + w.h : -1;
      }
    }
  };
  // Stage the warp's i-th list entry in stage sidx: lane 0 arms the stage's
  // mbarrier with the byte count, then each lane owning a valid page copies it.
  auto issue_int2 = [&](int i, int sidx) {
    walk_to(iw, ga + i);
    if (i % CPF == 0) fill_cache(i);
    const bool mine = lane / PPS == i % CPF;
    const bool ok = mine && rec >= 0;
    const unsigned okm = __ballot_sync(FULLM, ok);
    const unsigned badm = __ballot_sync(FULLM, mine && rec == -1);
    const uint32_t bits = (okm >> ((i % CPF) * PPS)) & ALL_PAGES;
    uint64_t* bar = &bars[warp][sidx];
    if (lane == 0) {
      if (badm) flag_error(err, ERR_BLOCK_RANGE);
      sflag[warp][sidx] = (uint8_t)bits;
      mbar_arrive_expect_tx(bar, (uint32_t)__popc(bits) * REC);
    }
    __syncwarp();
    if (ok) {
      fence_proxy_async();
      bulk_g2s(stage_ptr(warp, sidx) + (lane % PPS) * REC, pool + (size_t)rec * g.record, REC, bar);
    }
  };
  // Window record j of the warp's slice (one 4,096-byte copy by lane 0).
  // Local record r of a unit: sink record r (r < ns), else the recent group of
  // positions starting at (a & ~7) + 8 (r - ns), a = max(S_w, len - R_w).
  auto wrec_first_pos = [&](const ChunkWalker& w, int r) {
    const int ns = (min(S_w, w.len) + 7) >> 3;
    return r < ns ? 8 * r : (max(S_w, w.len - R_w) & ~7) + 8 * (r - ns);
  };
  auto issue_win = [&](int j, int sidx) {
    walk_w(iww, gaw + j);
    const int p0 = wrec_first_pos(iww, gaw + j - iww.S);
    const int slot = p0 < S_w ? p0 : S_w + (R_w ? p0 % R_w : 0);
    uint64_t* bar = &bars[warp][sidx];
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, WIN_REC_BYTES);
      fence_proxy_async();
      bulk_g2s(stage_ptr(warp, sidx),
               win.buf + (((size_t)iww.b * Hkv + iww.h) * n_wrec + slot / WIN_REC_TOKENS) * WIN_REC_BYTES,
               WIN_REC_BYTES, bar);
    }
    __syncwarp();
  };
  // Fill f of the warp's stage ring: even warps take their window records first,
  // odd warps last, so that window (bandwidth) and INT2 (instruction) phases overlap.
  const bool win_first = WIN && (gw & 1) == 0;
  auto issue = [&](int f) {
    n_issued = f + 1;
    const int sidx = f % NST;
    if (WIN && (win_first ? f < my_nw : f >= my_n)) issue_win(win_first ? f : f - my_n, sidx);
    else issue_int2(win_first ? f - my_nw : f, sidx);
  };

  // With a step's append (kvq_decode_step) the query preparation writes the new token
  // into the last page of every sequence (and, with windows, into the unit's last
  // window record): a warp whose first fills include the last entry of a unit in
  // either list issues them only after that kernel has completed.
  bool early = true;
  if (step_append && F > 0) {
    ChunkWalker w = iw, w2 = iww;
    for (int f = 0; f < NST && f < F; ++f) {
      if (WIN && (win_first ? f < my_nw : f >= my_n)) {
        const int j = win_first ? f : f - my_n;
        walk_w(w2, gaw + j);
        if (gaw + j == w2.E - 1) early = false;
      } else {
        const int i = WIN && win_first ? f - my_nw : f;
        walk_to(w, ga + i);
        if (ga + i == w.E - 1) early = false;
      }
    }
  }
  if (F > 0) {
    if (lane == 0) {
      for (int s = 0; s < NST; ++s) mbar_init(&bars[warp][s], 1);
      fence_mbar_init();
    }
    __syncwarp();
    if (early)
      for (int f = 0; f < NST && f < F; ++f) issue(f);
  }
  pdl_wait();               // the query fragments and spans come from qprep_kernel
  if (F > 0 && !early)
    for (int f = 0; f < NST && f < F; ++f) issue(f);
  pdl_launch_dependents();  // the combine kernel may be scheduled as blocks retire
  if (F <= 0) return;       // no block-level synchronisation follows

  // ---- per-segment state (one segment = the warp's entries of one unit) ----
  uint32_t bq[NT][8][2];  // B fragments of q'.c, k-slice s (see qprep_kernel)
  float dsc[NT], qsum_s[NT], tau_s[NT], m_s[NT], thr[NT], nm[NT], lp[NT], zp[NT];
  float acc[NT][8][4];
  int cur_u = -1, cur_S = 0, cur_E = 0;

  auto start_segment = [&](int u) {
    const uint32_t* fr = ws.qfrag + (size_t)u * NT * 16 * 32 + lane;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        bq[nt][s][0] = __ldg(fr + (nt * 16 + 2 * s) * 32);
        bq[nt][s][1] = __ldg(fr + (nt * 16 + 2 * s + 1) * 32);
      }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int j = 4 * nt + ti;
      const float4 c = j < G ? __ldg(reinterpret_cast<const float4*>(ws.qconst) + (size_t)u * G + j)
                             : make_float4(1.f, 0.f, TAU, 0.f);
      dsc[nt] = c.x;
      qsum_s[nt] = c.y;
      tau_s[nt] = c.z;
      m_s[nt] = -INFINITY;
      thr[nt] = -INFINITY;
      nm[nt] = 0.f;
      lp[nt] = 0.f;
      zp[nt] = 0.f;
#pragma unroll
      for (int f = 0; f < 8; ++f) acc[nt][f][0] = acc[nt][f][1] = acc[nt][f][2] = acc[nt][f][3] = 0.f;
    }
  };

  // Write the warp's partial of the open segment (slot gw + unit).
  auto finish_segment = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lp[nt] += __shfl_xor_sync(FULLM, lp[nt], o);
        zp[nt] += __shfl_xor_sync(FULLM, zp[nt], o);
      }
    }
    float* pp = ws.part + (size_t)(gw + cur_u) * G * PART;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int j = 4 * nt + ti;
      if (j < G) {
        float o[16];
#pragma unroll
        for (int f = 0; f < 8; ++f) {
          const float sc = (float)(1 << (24 - v_pe(f)));
          o[f] = fmaf(fmaf(acc[nt][f][1], LO_UNSCALE, acc[nt][f][0]), sc, zp[nt]);      // channel 8g + f
          o[8 + f] = fmaf(fmaf(acc[nt][f][3], LO_UNSCALE, acc[nt][f][2]), sc, zp[nt]);  // channel 64 + 8g + f
        }
        float4* dst = reinterpret_cast<float4*>(pp + j * PART);
        dst[2 * gi] = make_float4(o[0], o[1], o[2], o[3]);
        dst[2 * gi + 1] = make_float4(o[4], o[5], o[6], o[7]);
        dst[16 + 2 * gi] = make_float4(o[8], o[9], o[10], o[11]);
        dst[16 + 2 * gi + 1] = make_float4(o[12], o[13], o[14], o[15]);
        if (gi == 0) {
          pp[j * PART + D] = m_s[nt] * dsc[nt];
          pp[j * PART + D + 1] = lp[nt];
        }
      }
    }
    // the slice holding the unit's first entry records which slices meet the unit
    if (lane == 0 && gw == cur_S / Ww) ws.span[cur_u] = make_int2(gw, (cur_E - 1) / Ww);
  };

  const uint32_t sel = (gi & 1) ? 0x7632u : 0x5410u;  // pick remainder / high halves
  const int srcA = 8 * ti + (gi >> 1);                // lanes holding tokens 2t, 2t + 8 of head 4nt + g/2
  // ldmatrix row address of this lane inside a staged chunk (tile 0); tile 1 is 1,152 bytes on
  const uint32_t vrow = smem_u32(stage_ptr(warp, 0)) + CL::v(0, 8 * (lane >> 4) + (lane & 7)) + 16 * ((lane >> 3) & 1);

  // One 32-token chunk from a staged stage.  FULL: every token valid and copied.
  auto chunk = [&](auto full_tag, const uint8_t* st, uint32_t vaddr, int tok0, int len, int bits) {
    constexpr bool FULL = decltype(full_tag)::value;
    bool rok[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int u = k >> 1, r = gi + 8 * (k & 1);
      rok[k] = FULL || ((tok0 + 16 * u + r < len) && ((bits >> CL::page(u, r)) & 1));
    }
    // ---- scores (Eqs. 21-22): s (q'.c) + z sum(q'), rows g and g + 8 of each tile ----
    float sc[NT][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint2 kr0 = *reinterpret_cast<const uint2*>(st + CL::k(u, gi) + 8 * ti);
      const uint2 kr1 = *reinterpret_cast<const uint2*>(st + CL::k(u, gi + 8) + 8 * ti);
      float d[NT][4];
      const uint32_t s00 = kr0.x >> 10, s01 = kr0.y >> 10, s10 = kr1.x >> 10, s11 = kr1.y >> 10;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t mask = s <= 4 ? (0x00030003u << (2 * s)) : (0x00030003u << (2 * s - 10));
        const uint32_t a0 = (s <= 4 ? kr0.x : s00) & mask;  // row g,   channels 32t+s | 32t+8+s
        const uint32_t a1 = (s <= 4 ? kr1.x : s10) & mask;  // row g+8
        const uint32_t a2 = (s <= 4 ? kr0.y : s01) & mask;  // row g,   channels 32t+16+s | 32t+24+s
        const uint32_t a3 = (s <= 4 ? kr1.y : s11) & mask;  // row g+8
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (s == 0) mma16816_zero(d[nt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
          else mma16816(d[nt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
        }
      }
      const float2 km0 = meta_pair(st + CL::km(u, gi));
      const float2 km1 = meta_pair(st + CL::km(u, gi + 8));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float s0 = fmaf(km0.x, fmaf(d[nt][1], LO_UNSCALE, d[nt][0]), km0.y * qsum_s[nt]);
        const float s1 = fmaf(km1.x, fmaf(d[nt][3], LO_UNSCALE, d[nt][2]), km1.y * qsum_s[nt]);
        sc[nt][2 * u] = rok[2 * u] ? s0 : -INFINITY;
        sc[nt][2 * u + 1] = rok[2 * u + 1] ? s1 : -INFINITY;
      }
    }
    // value metadata: scale (negated in tile 1) and zero term z (+ 3 s in tile 1)
    float vsx[4], vzz[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 vm = meta_pair(st + CL::vm(k >> 1, gi + 8 * (k & 1)));
      vsx[k] = (k >> 1) ? -vm.x : vm.x;
      vzz[k] = (k >> 1) ? fmaf(3.f, vm.x, vm.y) : vm.y;
    }

    // ---- online softmax (Eq. 2) with lazy rescale, and the weights p_t s_t ----
    uint32_t bp[NT][2][2];  // [n-tile][tile][b register]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float lm = fmaxf(fmaxf(sc[nt][0], sc[nt][1]), fmaxf(sc[nt][2], sc[nt][3]));
      if (__any_sync(FULLM, lm > thr[nt])) {  // some head's maximum moved by > TAU
        float mx = fmaxf(lm, __shfl_xor_sync(FULLM, lm, 4));
        mx = fmaxf(mx, __shfl_xor_sync(FULLM, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(FULLM, mx, 16));
        const bool need = mx > thr[nt];
        const float alpha = need ? ex2((m_s[nt] - mx) * dsc[nt]) : 1.f;
        if (need) {
          m_s[nt] = mx;
          thr[nt] = mx + tau_s[nt];
          nm[nt] = -mx * dsc[nt];
        }
        lp[nt] *= alpha;
        zp[nt] *= alpha;
#pragma unroll
        for (int f = 0; f < 8; ++f) {
          acc[nt][f][0] *= alpha; acc[nt][f][1] *= alpha; acc[nt][f][2] *= alpha; acc[nt][f][3] *= alpha;
        }
      }
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float p = ex2(fmaf(sc[nt][k], dsc[nt], nm[nt]));
        float w = p * vsx[k];
        float pz = p * vzz[k];
        if (!FULL) {
          p = rok[k] ? p : 0.f;
          w = rok[k] ? w : 0.f;
          pz = rok[k] ? pz : 0.f;
        }
        lp[nt] += p;
        zp[nt] += pz;
        const float hf = half_rn(w);
        pk[k] = pack_half2(w, (w - hf) * LO_SCALE);  // low half: fp16(w); high half: remainder * 2^11
      }
      // B fragment of tile u: k = 2t, 2t+1, 2t+8, 2t+9 <-> tokens 2t, 2t+1, 2t+8, 2t+9;
      // column g <-> head 4nt + g/2, high part (g even) or remainder (g odd)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t y0 = __shfl_sync(FULLM, pk[2 * u], srcA);
        const uint32_t y1 = __shfl_sync(FULLM, pk[2 * u], srcA + 4);
        const uint32_t y2 = __shfl_sync(FULLM, pk[2 * u + 1], srcA);
        const uint32_t y3 = __shfl_sync(FULLM, pk[2 * u + 1], srcA + 4);
        bp[nt][u][0] = prmt(y0, y1, sel);
        bp[nt][u][1] = prmt(y2, y3, sel);
      }
    }

    // ---- values (Eq. 5): D[channel][2j + {hi,lo}] += 2^(pe-24) sum_t code_t (+-w_t) ----
    // Tile 0 enters as (c, +w) and tile 1 as (3 - c, -w), one logical operation
    // per two codes either way: the accumulated common part 1.5 (sum_tile0 w -
    // sum_tile1 w) cancels between neighbouring tiles instead of growing with the
    // context, and the 3 s_t of tile 1 is restored through the zero term.
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      uint32_t rw[4], sw[4];  // element g / 8+g of tokens (2t, 2t+1) and (2t+8, 2t+9); byte-swapped
      ldsm_x4_trans(vaddr + u * 1152, rw);
#pragma unroll
      for (int x = 0; x < 4; ++x) sw[x] = prmt(rw[x], rw[x], 0x2301u);
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        const uint32_t mask = 0x00030003u << v_pe(f);
        uint32_t a[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint32_t src = v_swapped(f) ? sw[x] : rw[x];
          a[x] = u ? (~src & mask) : (src & mask);  // tile 1: 3 - c
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt][f], a[0], a[1], a[2], a[3], bp[nt][u][0], bp[nt][u][1]);
      }
    }
  };

  if constexpr (!WIN) {
    // without windows the fills are the list entries: the plain loop
    bool aborted = false;
    int consumed = 0;
    for (int i = 0; i < my_n; ++i) {
      const int sidx = i % NST;
      bool ok = false;
      for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][sidx], (i / NST) & 1);
      ok = __all_sync(FULLM, ok);
      if (!ok) {
        if (lane == 0) flag_error(err, ERR_TIMEOUT);
        aborted = true;
        break;
      }
      consumed = i + 1;
      walk_to(cw, ga + i);
      const int u = cw.b * Hkv + cw.h;
      if (u != cur_u) {
        if (cur_u >= 0) finish_segment();
        start_segment(u);
        cur_u = u;
        cur_S = cw.S;
        cur_E = cw.E;
      }
      const int bits = sflag[warp][sidx];
      const int tokS = (ga + i - cw.S) * 64;
#pragma unroll 1
      for (int sub = 0; sub < 2; ++sub) {  // the stage's two 32-token chunks
        const int tok0 = tokS + 32 * sub;
        if (tok0 >= cw.len) break;
        const uint8_t* st = stage_ptr(warp, sidx) + sub * CHUNK;
        const uint32_t vaddr = vrow + sidx * STAGE + sub * CHUNK;
        const int cbits = (bits >> (sub * PPC)) & (int)CHUNK_PAGES;
        if (tok0 + 32 <= cw.len && cbits == (int)CHUNK_PAGES) chunk(std::true_type{}, st, vaddr, tok0, cw.len, cbits);
        else chunk(std::false_type{}, st, vaddr, tok0, cw.len, cbits);
      }
      __syncwarp();
      if (i + NST < my_n) issue(i + NST);
    }
    if (aborted) {
      // wait (bounded) for the copies still in flight before the stages go away;
      // the open segment is dropped (its unit's output is not written, the error flag is set)
      for (int i = consumed; i < n_issued; ++i) {
        bool ok = false;
        for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][i % NST], (i / NST) & 1);
      }
      return;
    }
    if (cur_u >= 0) finish_segment();
    return;
  } else {
  int consumed = 0;  // fills consumed
  // Bounded wait for fill f; false (error flag set) if its copies never completed.
  auto wait_fill = [&](int f) {
    bool ok = false;
    for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][f % NST], (f / NST) & 1);
    ok = __all_sync(FULLM, ok);
    if (!ok && lane == 0) flag_error(err, ERR_TIMEOUT);
    return ok;
  };

  // ---- window phase: 8-token BF16 records, fills f0 .. f0 + my_nw - 1 ----
  // Keys (centred, not rotated) meet the unrotated query; values are already in
  // the rotated basis.  Scores: A = the 8 key rows (rows 8-15 of the tile are
  // zero), B = the query fragments (bf16 high part and remainder per head);
  // values: A = the value rows transposed (ldmatrix .trans), k = the 8 tokens.
  // Rows are stored with the 16-byte chunk c of row r at c ^ r, so the 8 rows of
  // one ldmatrix come from 8 different bank groups.
  auto run_win = [&](int f0) {
    if constexpr (WIN) {
      uint32_t bw[NT][8][2];
      float wm[NT], wthr[NT], wl[NT];
      float wacc[NT][8][4];
      int wu = -1, wS = 0, wE = 0;
      auto wstart = [&](int u) {
        const uint32_t* fr = ws.wqfrag + (size_t)u * NT * 16 * 32 + lane;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            bw[nt][s][0] = __ldg(fr + (nt * 16 + 2 * s) * 32);
            bw[nt][s][1] = __ldg(fr + (nt * 16 + 2 * s + 1) * 32);
          }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          wm[nt] = -INFINITY;
          wthr[nt] = -INFINITY;
          wl[nt] = 0.f;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) wacc[nt][mt][0] = wacc[nt][mt][1] = wacc[nt][mt][2] = wacc[nt][mt][3] = 0.f;
        }
      };
      auto wfinish = [&]() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) wl[nt] += __shfl_xor_sync(FULLM, wl[nt], o);
        float* pp = ws.partw + (size_t)(gw + wu) * G * PART;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int j = 4 * nt + ti;
          if (j < G) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {  // channel rows 16 mt + g and 16 mt + 8 + g; high part + remainder
              pp[j * PART + 16 * mt + gi] = wacc[nt][mt][0] + wacc[nt][mt][1];
              pp[j * PART + 16 * mt + 8 + gi] = wacc[nt][mt][2] + wacc[nt][mt][3];
            }
            if (gi == 0) {
              pp[j * PART + D] = wm[nt];
              pp[j * PART + D + 1] = wl[nt];
            }
          }
        }
        if (lane == 0 && gw == wS / Wwn) ws.spanw[wu] = make_int2(gw, (wE - 1) / Wwn);
      };
      const uint32_t krow = (uint32_t)(lane & 7) * 256u;
      for (int j = 0; j < my_nw; ++j) {
        const int f = f0 + j;
        const int sidx = f % NST;
        if (!wait_fill(f)) return false;
        consumed = f + 1;
        walk_w(cww, gaw + j);
        const int u = cww.b * Hkv + cww.h;
        if (u != wu) {
          if (wu >= 0) wfinish();
          wstart(u);
          wu = u;
          wS = cww.S;
          wE = cww.E;
        }
        // rows holding window positions: p0 + r inside the sink [0, min(S_w, len)) or the recent part [a, len)
        const int p0 = wrec_first_pos(cww, gaw + j - cww.S);
        const int lo = p0 < S_w ? 0 : max(S_w, cww.len - R_w);
        const int hi = p0 < S_w ? min(S_w, cww.len) : cww.len;
        const int first = max(lo - p0, 0), last = min(hi - p0, 8);
        const unsigned vmask = (0xffu >> (8 - last)) & (0xffu << first) & 0xffu;
        const uint32_t sbase = smem_u32(stage_ptr(warp, sidx)) + krow;
        float d[NT][4];
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {  // k-slices 2 sp and 2 sp + 1 (channels 32 sp .. 32 sp + 31)
          uint32_t kr[4];
          ldsm_x4(sbase + ((uint32_t)((4 * sp + (lane >> 3)) ^ (lane & 7)) << 4), kr);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (sp == 0) mma16816_bf16_zero(d[nt], kr[0], 0u, kr[1], 0u, bw[nt][0][0], bw[nt][0][1]);
            else mma16816_bf16(d[nt], kr[0], 0u, kr[1], 0u, bw[nt][2 * sp][0], bw[nt][2 * sp][1]);
            mma16816_bf16(d[nt], kr[2], 0u, kr[3], 0u, bw[nt][2 * sp + 1][0], bw[nt][2 * sp + 1][1]);
          }
        }
        const bool tv = (vmask >> gi) & 1u;  // this lane's row (token gi) holds a window position
        uint32_t bpw[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float sc = tv ? d[nt][0] + d[nt][1] : -INFINITY;  // log2 units (q carries log2(e)/sqrt(128))
          if (__any_sync(FULLM, sc > wthr[nt])) {
            float mx = fmaxf(sc, __shfl_xor_sync(FULLM, sc, 4));
            mx = fmaxf(mx, __shfl_xor_sync(FULLM, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(FULLM, mx, 16));
            const bool need = mx > wthr[nt];
            const float alpha = need ? ex2(wm[nt] - mx) : 1.f;
            if (need) {
              wm[nt] = mx;
              wthr[nt] = mx + TAU;
            }
            wl[nt] *= alpha;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              wacc[nt][mt][0] *= alpha; wacc[nt][mt][1] *= alpha; wacc[nt][mt][2] *= alpha; wacc[nt][mt][3] *= alpha;
            }
          }
          const float pw = ex2(sc - wm[nt]);
          wl[nt] += pw;
          const __nv_bfloat16 ph = __float2bfloat16_rn(pw);
          const __nv_bfloat16 pr = __float2bfloat16_rn(pw - __bfloat162float(ph));
          const uint32_t pk = (uint32_t)__bfloat16_as_ushort(ph) | ((uint32_t)__bfloat16_as_ushort(pr) << 16);
          // B fragment: tokens 2t, 2t + 1 of column g (head 4 nt + g/2, high part or remainder)
          bpw[nt] = prmt(__shfl_sync(FULLM, pk, srcA), __shfl_sync(FULLM, pk, srcA + 4), sel);
        }
        // rows outside the window may hold stale or unwritten data: zero them (their weight is 0 already)
        const uint32_t tmask = vmask == 0xffu ? 0xffffffffu
                                              : ((((vmask >> (2 * ti)) & 1u) ? 0x0000ffffu : 0u) |
                                                 (((vmask >> (2 * ti + 1)) & 1u) ? 0xffff0000u : 0u));
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {  // channel tiles 2 qq and 2 qq + 1
          uint32_t vr[4];
          ldsm_x4_trans(sbase + 2048u + ((uint32_t)((4 * qq + (lane >> 3)) ^ (lane & 7)) << 4), vr);
#pragma unroll
          for (int x = 0; x < 4; ++x) vr[x] &= tmask;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma16816_bf16(wacc[nt][2 * qq], vr[0], vr[1], 0u, 0u, bpw[nt], 0u);
            mma16816_bf16(wacc[nt][2 * qq + 1], vr[2], vr[3], 0u, 0u, bpw[nt], 0u);
          }
        }
        __syncwarp();
        if (f + NST < F) issue(f + NST);
      }
      if (wu >= 0) wfinish();
    }
    return true;
  };

  bool ok = true;
  if (win_first) ok = run_win(0);
  if (ok) {
    // ---- INT2 phase: the warp's list entries, fills f0 .. f0 + my_n - 1 (the plain loop) ----
    const int f0 = win_first ? my_nw : 0;
    for (int i = 0; i < my_n; ++i) {
      const int f = f0 + i;
      const int sidx = f % NST;
      bool got = false;
      for (int it = 0; it < WAIT_LIMIT && !got; ++it) got = mbar_try_wait(&bars[warp][sidx], (f / NST) & 1);
      got = __all_sync(FULLM, got);
      if (!got) {
        if (lane == 0) flag_error(err, ERR_TIMEOUT);
        ok = false;
        break;
      }
      consumed = f + 1;
      walk_to(cw, ga + i);
      const int u = cw.b * Hkv + cw.h;
      if (u != cur_u) {
        if (cur_u >= 0) finish_segment();
        start_segment(u);
        cur_u = u;
        cur_S = cw.S;
        cur_E = cw.E;
      }
      const int bits = sflag[warp][sidx];
      const int e = cw.len - R_w;  // INT2 positions end here (the recent window follows)
      const int tokS = S_w + (ga + i - cw.S) * 64;
#pragma unroll 1
      for (int sub = 0; sub < 2; ++sub) {  // the stage's two 32-token chunks
        const int tok0 = tokS + 32 * sub;
        if (tok0 >= e) break;
        const uint8_t* st = stage_ptr(warp, sidx) + sub * CHUNK;
        const uint32_t vaddr = vrow + sidx * STAGE + sub * CHUNK;
        const int cbits = (bits >> (sub * PPC)) & (int)CHUNK_PAGES;
        if (tok0 + 32 <= e && cbits == (int)CHUNK_PAGES) chunk(std::true_type{}, st, vaddr, tok0, e, cbits);
        else chunk(std::false_type{}, st, vaddr, tok0, e, cbits);
      }
      __syncwarp();
      if (f + NST < F) issue(f + NST);
    }
    if (ok && cur_u >= 0) finish_segment();
  }
  if (ok && !win_first) ok = run_win(my_n);
  if (!ok) {
    // wait (bounded) for the copies still in flight before the stages go away;
    // the open segment is dropped (its unit's output is not written, the error flag is set)
    for (int f = consumed; f < n_issued; ++f) {
      bool done = false;
      for (int it = 0; it < WAIT_LIMIT && !done; ++it) done = mbar_try_wait(&bars[warp][f % NST], (f / NST) & 1);
    }
  }
  }
}

// ---------------------------------------------------------------------------
// Combine: grid (U, G), nw warps (1..32, from the average partials per unit).
// o_rot of query head j of unit u is the log-sum-exp merge of the unit's
// partials (slots k + u, k0 <= k <= k1) in one pass: warp w folds the slots
// w, w + nw, ... (four at a time, their loads in flight together) into a running
// state (M, L, A) rescaled when the maximum moves, and the warp states are merged
// in warp order, so the result does not depend on timing.
// ---------------------------------------------------------------------------
constexpr int CB_MAX_WARPS = 32;

template <int G>
__global__ void __launch_bounds__(CB_MAX_WARPS * 32) decode_combine_kernel(int n_kv_heads, int n_q_heads, DecWs ws,
                                                                           float* __restrict__ o_rot) {
  __shared__ float sm_m[CB_MAX_WARPS], sm_l[CB_MAX_WARPS];
  __shared__ __align__(16) float sm_a[CB_MAX_WARPS][D];
  pdl_launch_dependents();  // a following projection may start streaming its (static) weights
  pdl_wait();               // the partials come from decode_split_kernel
  const int u = blockIdx.x, j = blockIdx.y;
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int2 sp = __ldcg(ws.span + u);
  if (sp.x > sp.y) return;  // no cached tokens (o = 0 already) or an invalid length
  const int ns = sp.y - sp.x + 1;
  const size_t stride = (size_t)G * PART;  // floats between consecutive slots
  const float* base = ws.part + ((size_t)(sp.x + u) * G + j) * PART;
  float M = -INFINITY, l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t0 = warp; t0 < ns; t0 += 4 * nw) {
    float2 ml[4];
    float4 x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = t0 + k * nw;
      ml[k] = make_float2(-INFINITY, 0.f);
      x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < ns) {
        ml[k] = __ldcg(reinterpret_cast<const float2*>(base + t * stride + D));
        x[k] = __ldcg(reinterpret_cast<const float4*>(base + t * stride) + lane);
      }
    }
    const float mn = fmaxf(fmaxf(M, fmaxf(ml[0].x, ml[1].x)), fmaxf(ml[2].x, ml[3].x));
    if (mn == -INFINITY) continue;  // nothing valid yet (uniform across the warp)
    const float r = M == -INFINITY ? 0.f : exp2f(M - mn);
    l *= r;
    a.x *= r; a.y *= r; a.z *= r; a.w *= r;
    M = mn;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float e = ml[k].x == -INFINITY ? 0.f : exp2f(ml[k].x - M);
      l = fmaf(e, ml[k].y, l);
      a.x = fmaf(e, x[k].x, a.x); a.y = fmaf(e, x[k].y, a.y); a.z = fmaf(e, x[k].z, a.z); a.w = fmaf(e, x[k].w, a.w);
    }
  }
  const int b = u / n_kv_heads, h = u % n_kv_heads;
  float4* dst = reinterpret_cast<float4*>(o_rot + ((size_t)b * n_q_heads + h * G + j) * D);
  if (nw == 1) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    dst[lane] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    return;
  }
  if (lane == 0) {
    sm_m[warp] = M;
    sm_l[warp] = l;
  }
  reinterpret_cast<float4*>(sm_a[warp])[lane] = a;
  __syncthreads();
  float Mt = -INFINITY;
  for (int w = 0; w < nw; ++w) Mt = fmaxf(Mt, sm_m[w]);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {  // 64 or more threads
    float A = 0.f, L = 0.f;
    if (Mt != -INFINITY)
      for (int w = 0; w < nw; ++w) {
        const float e = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - Mt);
        A = fmaf(e, sm_a[w][c], A);
        L = fmaf(e, sm_l[w], L);
      }
    o_rot[((size_t)b * n_q_heads + h * G + j) * D + c] = L > 0.f ? A / L : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Combine with BF16 windows: one CTA (8 warps) per (unit, query head j).  Warp w
// merges the slots w, w + 8, ... of the unit -- its INT2 partials, then its
// window partials -- in one online pass (running maximum, rescaled sums, several
// slots' loads in flight) into l, A (INT2, already in the rotated-V basis) and W
// (window values, unrotated); the warp states are merged in warp order
// (deterministic).  W is then rotated by R_V,h (Eq. 27): the FWHT for the signed
// Hadamard, and for a dense R each warp multiplies 16 rows of R, the row blocks
// added in warp order.
//   o_rot = (A + W R_V) / l
// ---------------------------------------------------------------------------
constexpr int CBW_WARPS = 8;

template <int G>
__global__ void __launch_bounds__(CBW_WARPS * 32) decode_combine_win_kernel(int n_kv_heads, int n_q_heads, DecWs ws,
                                                                           RotDev rot_v, float* __restrict__ o_rot) {
  __shared__ __align__(16) float sA[D];
  __shared__ __align__(16) float sW[D];
  __shared__ __align__(16) float sY[D];
  __shared__ float sL, sM;
  pdl_launch_dependents();  // a following projection may start streaming its (static) weights
  pdl_wait();               // the partials come from decode_split_kernel
  const int u = blockIdx.x, j = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = u / n_kv_heads, h = u % n_kv_heads;
  const int2 sp = __ldcg(ws.span + u), spw = __ldcg(ws.spanw + u);
  const int ni = max(0, sp.y - sp.x + 1), nwin = max(0, spw.y - spw.x + 1);
  const int ns = ni + nwin;
  if (ns == 0) return;  // no cached tokens (o = 0 already) or an invalid length
  const size_t stride = (size_t)G * PART;
  const float* base = ws.part + ((size_t)(sp.x + u) * G + j) * PART;
  const float* basew = nwin ? ws.partw + ((size_t)(spw.x + u) * G + j) * PART : base;

  float m = -INFINITY, l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), w = a;
#pragma unroll 4
  for (int t = warp; t < ns; t += CBW_WARPS) {
    const bool win = t >= ni;
    const float* pp = win ? basew + (t - ni) * stride : base + t * stride;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(pp + D));
    const float4 x = __ldcg(reinterpret_cast<const float4*>(pp) + lane);
    const float mn = fmaxf(m, ml.x);
    const float so = m == -INFINITY ? 0.f : exp2f(m - mn);  // rescale of the running sums
    const float e = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mn);
    const float ea = win ? 0.f : e, ew = win ? e : 0.f;
    m = mn;
    l = fmaf(e, ml.y, l * so);
    a.x = fmaf(ea, x.x, a.x * so); a.y = fmaf(ea, x.y, a.y * so);
    a.z = fmaf(ea, x.z, a.z * so); a.w = fmaf(ea, x.w, a.w * so);
    w.x = fmaf(ew, x.x, w.x * so); w.y = fmaf(ew, x.y, w.y * so);
    w.z = fmaf(ew, x.z, w.z * so); w.w = fmaf(ew, x.w, w.w * so);
  }
  // warp states merged in warp order, rescaled to the running maximum
  for (int wv = 0; wv < CBW_WARPS; ++wv) {
    if (warp == wv) {
      const float m0 = wv ? sM : -INFINITY;
      const float mn = fmaxf(m0, m);
      const float s0 = m0 == -INFINITY ? 0.f : exp2f(m0 - mn);
      const float s1 = m == -INFINITY ? 0.f : exp2f(m - mn);
      float4 A = wv ? reinterpret_cast<float4*>(sA)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      float4 W = wv ? reinterpret_cast<float4*>(sW)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      A.x = fmaf(s1, a.x, A.x * s0); A.y = fmaf(s1, a.y, A.y * s0);
      A.z = fmaf(s1, a.z, A.z * s0); A.w = fmaf(s1, a.w, A.w * s0);
      W.x = fmaf(s1, w.x, W.x * s0); W.y = fmaf(s1, w.y, W.y * s0);
      W.z = fmaf(s1, w.z, W.z * s0); W.w = fmaf(s1, w.w, W.w * s0);
      reinterpret_cast<float4*>(sA)[lane] = A;
      reinterpret_cast<float4*>(sW)[lane] = W;
      __syncwarp();
      if (lane == 0) {
        sL = fmaf(s1, l, (wv ? sL : 0.f) * s0);
        sM = mn;
      }
    }
    __syncthreads();
  }
  // rotate the window sum: y = W R_V,h
  if (rot_v.kind == KVQ_ROT_DENSE) {
    // warp w: rows 16 w .. 16 w + 15 of R (input channels), lane: output channels 4 lane .. 4 lane + 3
    const float4* R = reinterpret_cast<const float4*>(rot_v.dense + (size_t)h * D * D) + lane;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float4 r = __ldg(R + (size_t)(16 * warp + c) * (D / 4));
      const float x = sW[16 * warp + c];
      y.x = fmaf(x, r.x, y.x); y.y = fmaf(x, r.y, y.y); y.z = fmaf(x, r.z, y.z); y.w = fmaf(x, r.w, y.w);
    }
    for (int wv = 0; wv < CBW_WARPS; ++wv) {  // row blocks added in warp order
      if (warp == wv) {
        float4 s4 = wv ? reinterpret_cast<float4*>(sY)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        s4.x += y.x; s4.y += y.y; s4.z += y.z; s4.w += y.w;
        reinterpret_cast<float4*>(sY)[lane] = s4;
      }
      __syncthreads();
    }
  } else {
    if (warp == 0) {
      float4 x = reinterpret_cast<const float4*>(sW)[lane];
      if (rot_v.kind == KVQ_ROT_SIGNED_HADAMARD) x = rotate_vec_warp(x, rot_v, h, lane, false);
      reinterpret_cast<float4*>(sY)[lane] = x;
    }
    __syncthreads();
  }
  if (threadIdx.x < D) {
    const int c = threadIdx.x;
    o_rot[((size_t)b * n_q_heads + h * G + j) * D + c] = sL > 0.f ? (sA[c] + sY[c]) / sL : 0.f;
  }
}

// Shared-memory ring of the decode kernel: per warp DEC_STAGES stages of 64 tokens.
constexpr int DEC_WARP_SMEM = DEC_STAGES * 2 * 1152 * 2;

template <int G, int P, bool WIN>
cudaError_t decode_smem_attr() {
  static std::atomic<unsigned long long> done{0};  // one set of per-device flags per kernel instance
  return smem_limit_once(done, decode_split_kernel<G, P, WIN>, dec_max_warps(G) * DEC_WARP_SMEM);
}

cudaError_t launch_decode(const PageGeom& g, int n_q_heads, int n_seqs, const void* q, int q_dtype,
                          const int32_t* seq_lens, int max_seq_len, const int32_t* table, RotDev rot_k,
                          const uint8_t* pool, int n_ctas, void* ws_base, float* o_rot, unsigned* err,
                          cudaStream_t s, WinGeom win, RotDev rot_v, const StepAppend* app) {
  (void)max_seq_len;
  if (n_seqs == 0) return cudaSuccess;
  const int gqa = n_q_heads / g.n_kv_heads;
  const bool windows = win.sink + win.recent > 0;
  if (app && (app->win.sink != win.sink || app->win.recent != win.recent || app->win.buf != win.buf))
    return cudaErrorInvalidValue;  // the step writes the windows the decode reads
  DecWs ws;
  decode_ws_layout(ws_base, n_seqs, g.n_kv_heads, gqa, n_ctas, windows, &ws);
  // query preparation: several sequences of a KV head per CTA when the batch has more units
  // than fit in one wave of it (two CTAs per SM), so R_K / R_V are loaded once per CTA
  const int qp_cap = 2 * device_sm_count();
  const int qp_spc = max(1, min(8, (n_seqs * g.n_kv_heads + qp_cap - 1) / qp_cap));
  const dim3 qg(g.n_kv_heads, (n_seqs + qp_spc - 1) / qp_spc);
  const bool dense = rot_k.kind == KVQ_ROT_DENSE;
  const StepAppend sa = app ? *app
                            : StepAppend{nullptr, nullptr, 0, RotDev{0, nullptr, nullptr}, nullptr, 1.f, 1.f, nullptr,
                                         WinGeom{0, 0, nullptr}, nullptr};
  const int qpa_smem = qpa_smem_bytes(app && app->rot_v.kind == KVQ_ROT_DENSE);
#define KVQ_QPREP_AW(GG, DD, WW)                                                                              \
  do {                                                                                                        \
    static std::atomic<unsigned long long> attr{0};                                                          \
    const cudaError_t ea = smem_limit_once(attr, qprep_kernel<GG, DD, true, WW>, qpa_smem_bytes(true));       \
    if (ea != cudaSuccess) return ea;                                                                         \
    qprep_kernel<GG, DD, true, WW><<<qg, QP_THREADS, qpa_smem, s>>>(n_q_heads, g.n_kv_heads, q, q_dtype, rot_k, \
                                                                   seq_lens, ws, o_rot, g, table, sa, err, n_seqs, \
                                                                   qp_spc);                                   \
  } while (0)
#define KVQ_QPREP_A(GG, DD)                                                                                   \
  if (app && windows) KVQ_QPREP_AW(GG, DD, true);                                                             \
  else if (app) KVQ_QPREP_AW(GG, DD, false);                                                                  \
  else qprep_kernel<GG, DD, false><<<qg, QP_THREADS, 0, s>>>(n_q_heads, g.n_kv_heads, q, q_dtype, rot_k,       \
                                                            seq_lens, ws, o_rot, g, table, sa, err, n_seqs, qp_spc)
#define KVQ_QPREP(GG) \
  if (dense) { KVQ_QPREP_A(GG, true); } else { KVQ_QPREP_A(GG, false); }
  switch (gqa) {
    case 1: KVQ_QPREP(1); break;
    case 2: KVQ_QPREP(2); break;
    case 4: KVQ_QPREP(4); break;
    case 8: KVQ_QPREP(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_QPREP
#undef KVQ_QPREP_A
#undef KVQ_QPREP_AW
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // The decode kernel is a programmatic dependent of qprep_kernel.  Its 4 * n_ctas
  // warps run as one block per SM when they fill every SM with a full set of
  // partitions.  With the step's append, the query preparation holds tens of KB of
  // shared memory per block while it runs, so the warps of an SM come as two blocks:
  // the first fits beside a query-preparation block and stages its first copies
  // while the append still runs.
  const int n_sm = device_sm_count();
  const bool per_sm = n_ctas == n_sm * ctas_per_sm(gqa);
  const int dnw = !per_sm ? DEC_WARPS : app ? dec_max_warps(gqa) / 2 : dec_max_warps(gqa);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(DEC_WARPS * n_ctas / dnw);
  cfg.blockDim = dim3(32 * dnw);
  cfg.dynamicSmemBytes = dnw * DEC_WARP_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define KVQ_DEC_W(GG, PP, WW)                                                                              \
  do {                                                                                                    \
    e = decode_smem_attr<GG, PP, WW>();                                                                   \
    if (e == cudaSuccess)                                                                                 \
      e = cudaLaunchKernelEx(&cfg, decode_split_kernel<GG, PP, WW>, g, n_seqs, n_q_heads, seq_lens, table, pool, \
                             ws, o_rot, err, win, app ? 1 : 0);                                            \
  } while (0)
#define KVQ_DEC(GG, PP) \
  if (windows) KVQ_DEC_W(GG, PP, true); else KVQ_DEC_W(GG, PP, false)
#define KVQ_DEC_P(GG) \
  if (g.page_tokens == 16) { KVQ_DEC(GG, 16); } else { KVQ_DEC(GG, 8); }
  switch (gqa) {
    case 1: KVQ_DEC_P(1); break;
    case 2: KVQ_DEC_P(2); break;
    case 4: KVQ_DEC_P(4); break;
    case 8: KVQ_DEC_P(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_DEC_P
#undef KVQ_DEC
#undef KVQ_DEC_W
  if (e != cudaSuccess) return e;

  // the combine is a programmatic dependent of the decode kernel
  // warps per (unit, head): ~8 partials each, 1 .. 32
  const int units = n_seqs * g.n_kv_heads;
  const int per_unit = (DEC_WARPS * n_ctas + units - 1) / units + 1;
  int nw = 1;
  while (nw < CB_MAX_WARPS && nw * 8 < per_unit) nw *= 2;
  cfg.gridDim = dim3(units, gqa);
  cfg.blockDim = dim3(windows ? CBW_WARPS * 32 : nw * 32);
  cfg.dynamicSmemBytes = 0;
#define KVQ_CB(GG)                                                                                          \
  e = windows ? cudaLaunchKernelEx(&cfg, decode_combine_win_kernel<GG>, g.n_kv_heads, n_q_heads, ws, rot_v, o_rot) \
              : cudaLaunchKernelEx(&cfg, decode_combine_kernel<GG>, g.n_kv_heads, n_q_heads, ws, o_rot)
  switch (gqa) {
    case 1: KVQ_CB(1); break;
    case 2: KVQ_CB(2); break;
    case 4: KVQ_CB(4); break;
    case 8: KVQ_CB(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_CB
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
