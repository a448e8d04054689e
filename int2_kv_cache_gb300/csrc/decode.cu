// Read path: split-K decode attention straight off the packed INT2 pages, and
// the log-sum-exp combine of the split partials.
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
// Kernel structure (one CTA = one (sequence, KV head, split), 4 warps):
// * each warp owns every 4th 32-token chunk of the split and streams its
//   chunks through a ring of shared-memory stages with cp.async.bulk copies
//   completed on mbarriers (two 1,152-byte page records per stage for 16-token
//   pages, four 576-byte records for 8-token pages), one page per lane;
// * q'.c and sum_t (p_t s_t) c_t are warp-level tensor-core products
//   (mma.sync m16n8k16, fp16 inputs, fp32 accumulation).  A 2-bit field masked
//   in place inside a 16-bit word is the fp16 value c * 2^(p-24) (a subnormal,
//   p = the field's bit offset), so the operands need one logical operation per
//   two codes, and the power-of-two factor is compensated exactly in the other
//   operand.  The value codes are read transposed (ldmatrix .trans) so that
//   each register holds two tokens of one channel group, as the product wants.
//   The fp32 operand of each product (the rotated query, the weights p_t s_t)
//   is split into an fp16 high part and an fp16 remainder occupying the two
//   MMA columns of one head, which keeps ~22 significant bits;
// * the softmax runs online in base 2 per warp with a lazy reference maximum;
//   the four warps are merged in shared memory and the split's partial
//   (m, l, unnormalised acc) is written.
// A second kernel merges the splits.
#include <type_traits>

#include "quant_common.cuh"

namespace kvq {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int DEC_WARPS = 4;
constexpr int DEC_STAGES = 4;
constexpr unsigned ERR_TIMEOUT = 8u;
constexpr uint32_t WAIT_HINT_NS = 100000;  // per try_wait: sleep up to 100 us
constexpr int WAIT_LIMIT = 20000;          // then give up (>= 2 s): error flag, no hang
// Lazy softmax rescaling: the running sums keep their reference maximum until a
// tile's maximum exceeds it by more than TAU (log2 units), so weights stay <= 2^TAU.
constexpr float TAU = 6.f;
// The fp16 remainder column carries (x - fp16(x)) * 2^11, keeping it out of the
// subnormal range whenever the high part is normal.
constexpr float LO_SCALE = 2048.f;
constexpr float LO_UNSCALE = 1.f / 2048.f;

struct Partials {
  float* acc;  // [B][Hq][S][128]
  float* ml;   // [B][Hq][S][2]: running max (log2 units), sum
};

__host__ __device__ inline Partials partials_from_ws(void* ws, int n_seqs, int n_q_heads, int n_splits) {
  Partials p;
  p.acc = static_cast<float*>(ws);
  p.ml = p.acc + (size_t)n_seqs * n_q_heads * n_splits * D;
  return p;
}

// Workspace: partials acc [B][Hq][S][128], (m, l) [B][Hq][S][2], then the rotated,
// pre-scaled queries q' [B][Hq][128] (fp32).
__host__ __device__ inline float* rotated_q_from_ws(void* ws, int n_seqs, int n_q_heads, int n_splits) {
  return static_cast<float*>(ws) + (size_t)n_seqs * n_q_heads * n_splits * (D + 2);
}

size_t decode_workspace_bytes(int n_seqs, int n_q_heads, int n_splits) {
  return (size_t)n_seqs * n_q_heads * (n_splits * (D + 2) + D) * sizeof(float);
}

int decode_auto_splits(int n_seqs, int n_kv_heads, int max_seq_len, int page_tokens) {
  (void)page_tokens;
  const int chunks = (max_seq_len + 31) / 32;
  const long long units = (long long)n_seqs * n_kv_heads;
  const int target = 152 * 4;
  int s = (int)((target + units - 1) / units);
  const int cap = chunks / 8 > 1 ? chunks / 8 : 1;  // keep >= 8 chunks (2 per warp) per split
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  if (s > 256) s = 256;
  return s;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Waits (suspended, up to the time hint) for the phase with the given parity.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(WAIT_HINT_NS)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

__device__ __forceinline__ float2 meta_pair(const uint8_t* p) {
  const uint32_t m = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(__half2float(__ushort_as_half((unsigned short)(m & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(m >> 16))));
}

// Value codes are read with a transposing shared-memory load (ldmatrix .trans):
// each register then holds one 16-bit element (8 channels) of two consecutive
// tokens.  Field f (channel 8e + f) is masked in place for f = 1..4 (bit 2f)
// and from the byte-swapped word for f = 0, 5, 6, 7 (bits 8, 2, 4, 6), so its
// fp16 value is c * 2^(pe-24) with pe in {2, 4, 6, 8}.
__host__ __device__ constexpr int v_pe(int f) { return f == 0 ? 8 : (f <= 4 ? 2 * f : 2 * f - 8); }
__host__ __device__ constexpr bool v_swapped(int f) { return f == 0 || f >= 5; }

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// ---------------------------------------------------------------------------
// Query rotation (Eq. 22): q'[b][j] = q[b][j] R_K,h(j) * log2(e)/sqrt(128), once
// per decode call.  grid = (n_kv_heads, ceil(n_seqs / QP_SEQS)), block = 256.
// A dense R_h is staged in shared memory; thread (d, half) produces channel d
// of every other query vector of the CTA.
// ---------------------------------------------------------------------------
constexpr int QP_SEQS = 4;

template <bool DENSE>
__global__ void __launch_bounds__(256) qprep_kernel(int n_seqs, int n_q_heads, int gqa,
                                                    const void* __restrict__ q, int q_dtype, RotDev rot,
                                                    float* __restrict__ qr) {
  extern __shared__ float sm[];  // dense: R [128][128], then q vectors [QP_SEQS * gqa][128]
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * QP_SEQS;
  const int nb = min(QP_SEQS, n_seqs - b0);
  const int nv = nb * gqa;
  const float sc = LOG2E * INV_SQRT_D;
  if (DENSE) {
    float* Rs = sm;
    float* qv = sm + D * D;
    const float4* src = reinterpret_cast<const float4*>(rot.dense + (size_t)h * D * D);
    for (int i = threadIdx.x; i < D * D / 4; i += 256) reinterpret_cast<float4*>(Rs)[i] = __ldg(src + i);
    for (int i = threadIdx.x; i < nv * D; i += 256) {
      const int v = i / D, c = i % D;
      const int b = b0 + v / gqa, j = h * gqa + v % gqa;
      qv[i] = load1(q, ((size_t)b * n_q_heads + j) * D + c, q_dtype);
    }
    __syncthreads();
    const int d = threadIdx.x & 127, half = threadIdx.x >> 7;
    for (int v = half; v < nv; v += 2) {
      const float* x = qv + v * D;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; c += 4) {
        a0 = fmaf(x[c], Rs[c * D + d], a0);
        a1 = fmaf(x[c + 1], Rs[(c + 1) * D + d], a1);
        a2 = fmaf(x[c + 2], Rs[(c + 2) * D + d], a2);
        a3 = fmaf(x[c + 3], Rs[(c + 3) * D + d], a3);
      }
      const int b = b0 + v / gqa, j = h * gqa + v % gqa;
      qr[((size_t)b * n_q_heads + j) * D + d] = ((a0 + a1) + (a2 + a3)) * sc;
    }
  } else {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int v = warp; v < nv; v += 8) {
      const int b = b0 + v / gqa, j = h * gqa + v % gqa;
      float4 x = load4(q, ((size_t)b * n_q_heads + j) * D + 4 * lane, q_dtype);
      x = rotate_vec_warp(x, rot, h, lane, false);
      x.x *= sc; x.y *= sc; x.z *= sc; x.w *= sc;
      reinterpret_cast<float4*>(qr + ((size_t)b * n_q_heads + j) * D)[lane] = x;
    }
  }
}

// ---------------------------------------------------------------------------
// The split kernel.  grid = (n_splits, n_kv_heads, n_seqs), block = 128.
// G = query heads per KV head; NT = n-tiles of 8 columns (2 columns per head).
// A split is a range of 32-token chunks; warp w takes chunks w, w + 4, ...
//
// Scores are kept per lane in units of 1/dscale_j (dscale_j = 2^(16 + e_j), the
// power of two that undoes the query prescale), so they come out of the
// products with one multiply-add; the softmax exponent applies dscale_j.
//
// Centring of the value codes: tile 0 of a chunk enters as (c, +w) and tile 1
// as (3 - c, -w), one logical operation per two codes either way.  The tensor
// cores then accumulate sum_t w_t c_t - 3 sum_{t in tile 1} w_t, whose common
// part 1.5 (sum_tile0 w - sum_tile1 w) cancels between neighbouring tiles
// instead of growing with the context; 3 s_t is added back through the zero term.
// ---------------------------------------------------------------------------
template <int G, int P>
__global__ void __launch_bounds__(128, (G >= 8 ? 3 : 5)) decode_split_kernel(
    PageGeom g, int n_q_heads, const float* __restrict__ qr,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ table,
    const uint8_t* __restrict__ pool, int n_splits, Partials part, unsigned* err) {
  constexpr int NT = (G + 3) / 4;
  constexpr int PPC = 32 / P;       // pages per chunk
  constexpr int REC = 72 * P;       // bytes per page record
  constexpr int CHUNK = PPC * REC;  // 2304
  constexpr int CPF = 32 / PPC;     // chunks per fill of the page-id cache
  constexpr uint32_t ALL_PAGES = (1u << PPC) - 1u;
  constexpr unsigned FULLM = 0xffffffffu;
  using CL = ChunkLayout<P>;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;  // MMA group id, thread id in group

  __shared__ __align__(128) uint8_t stage[DEC_WARPS][DEC_STAGES][CHUNK];
  __shared__ __align__(8) uint64_t bars[DEC_WARPS][DEC_STAGES];
  __shared__ __align__(16) float qs[G][D];
  __shared__ float qsum[G], qexp[G];
  __shared__ float sm_m[DEC_WARPS][G], sm_l[DEC_WARPS][G];
  __shared__ uint8_t sflag[DEC_WARPS][DEC_STAGES];  // bit p: page p of the chunk was copied

  int len = __ldg(seq_lens + b);
  if (len < 0 || len > g.max_blocks * g.page_tokens) {
    if (threadIdx.x == 0) flag_error(err, ERR_SEQ_RANGE);
    len = 0;
  }
  const int n_pages = (len + P - 1) / P;
  const int n_chunks = (len + 31) / 32;
  const int cps = (n_chunks + n_splits - 1) / n_splits;
  const int c_begin = split * cps;
  const int c_end = min(n_chunks, c_begin + cps);
  const int my_chunks = c_end > c_begin + warp ? (c_end - c_begin - warp + DEC_WARPS - 1) / DEC_WARPS : 0;
  const int32_t* trow = table + (size_t)b * g.max_blocks;
  const uint8_t* hbase = pool + (size_t)h * g.record;
  const size_t bstride = (size_t)g.n_kv_heads * g.record;

  // Page-id cache: lane l holds page l % PPC of the warp's chunk i0 + l / PPC;
  // -2 marks a page past the end of the sequence.
  int pid = -2;
  auto fill_cache = [&](int i0) {
    const int i = i0 + lane / PPC;
    const int pg = (c_begin + warp + DEC_WARPS * i) * PPC + lane % PPC;
    pid = (i < my_chunks && pg < n_pages) ? __ldg(trow + pg) : -2;
  };
  // Stage the warp's i-th chunk: lane 0 arms the stage's mbarrier with the byte
  // count, then each lane owning a valid page copies it.  Whole warp.
  auto issue = [&](int i) {
    if (i % CPF == 0 && i > 0) fill_cache(i);
    const int sidx = i % DEC_STAGES;
    const bool mine = lane / PPC == i % CPF;
    const bool ok = mine && pid >= 0 && pid < g.num_blocks;
    const unsigned okm = __ballot_sync(FULLM, ok);
    const unsigned badm = __ballot_sync(FULLM, mine && pid != -2 && !ok);
    const uint32_t bits = (okm >> ((i % CPF) * PPC)) & ALL_PAGES;
    uint64_t* bar = &bars[warp][sidx];
    if (lane == 0) {
      if (badm) flag_error(err, ERR_BLOCK_RANGE);
      sflag[warp][sidx] = (uint8_t)bits;
      mbar_arrive_expect_tx(bar, (uint32_t)__popc(bits) * REC);
    }
    __syncwarp();
    if (ok) {
      fence_proxy_async();
      bulk_g2s(stage[warp][sidx] + (lane % PPC) * REC, hbase + (size_t)pid * bstride, REC, bar);
    }
  };

  if (lane == 0) {
    for (int s = 0; s < DEC_STAGES; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  fill_cache(0);
  for (int i = 0; i < DEC_STAGES && i < my_chunks; ++i) issue(i);

  // ---- prologue: the rotated, pre-scaled queries q'_j (Eq. 22, from qprep_kernel) ----
  for (int jj = warp; jj < G; jj += DEC_WARPS) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(qr + ((size_t)b * n_q_heads + h * G + jj) * D) + lane);
    reinterpret_cast<float4*>(qs[jj])[lane] = v;
    const float tot = warp_sum(v.x + v.y + v.z + v.w);
    const float mx = warp_max(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    if (lane == 0) {
      qsum[jj] = tot;
      // power-of-two prescale keeping 256 * |q'| well inside the fp16 range
      int e = 0;
      while (e < 64 && mx * 256.f > 16384.f * exp2f((float)e)) ++e;
      qexp[jj] = (float)e;
    }
  }
  __syncthreads();

  // B fragments of q'.c: k-slice s uses the 2-bit field at bit p = 2s of each
  // 16-bit half of the key words; its fp16 value is c * 2^(pe-24) with
  // pe = p (p <= 8) or p - 10 (read after a 10-bit shift).  Column 2j holds the
  // fp16 high part of q'_j * 2^(8-pe-e_j), column 2j+1 the remainder * 2^11.
  uint32_t bq[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int j = 4 * nt + (gi >> 1);
    const bool lo_part = gi & 1;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int pe = s <= 4 ? 2 * s : 2 * s - 10;
      float vals[4] = {0.f, 0.f, 0.f, 0.f};
      if (j < G) {
        const float f = exp2f((float)(8 - pe) - qexp[j]);
        const int ch[4] = {32 * ti + s, 32 * ti + 8 + s, 32 * ti + 16 + s, 32 * ti + 24 + s};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float x = qs[j][ch[u]] * f;
          const float hi = half_rn(x);
          vals[u] = lo_part ? (x - hi) * LO_SCALE : hi;
        }
      }
      bq[nt][s][0] = pack_half2(vals[0], vals[1]);
      bq[nt][s][1] = pack_half2(vals[2], vals[3]);
    }
  }
  // Per-lane softmax state of head 4nt + ti, scores in units of 1/dsc.
  float dsc[NT], qsum_s[NT], tau_s[NT], m_s[NT], thr[NT], nm[NT], lp[NT], zp[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int j = 4 * nt + ti;
    dsc[nt] = j < G ? exp2f(16.f + qexp[j]) : 1.f;
    qsum_s[nt] = j < G ? qsum[j] * exp2f(-16.f - qexp[j]) : 0.f;
    tau_s[nt] = TAU / dsc[nt];
    m_s[nt] = -INFINITY;
    thr[nt] = -INFINITY;
    nm[nt] = 0.f;
    lp[nt] = 0.f;
    zp[nt] = 0.f;
  }
  const uint32_t sel = (gi & 1) ? 0x7632u : 0x5410u;  // pick remainder / high halves
  const int srcA = 8 * ti + (gi >> 1);                // lanes holding tokens 2t, 2t + 8 of head 4nt + g/2
  // ldmatrix row address of this lane inside a staged chunk (tile 0); tile 1 is 1,152 bytes on
  const uint32_t vrow = smem_u32(stage[warp][0]) + CL::v(0, 8 * (lane >> 4) + (lane & 7)) + 16 * ((lane >> 3) & 1);

  float acc[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int f = 0; f < 8; ++f) acc[nt][f][0] = acc[nt][f][1] = acc[nt][f][2] = acc[nt][f][3] = 0.f;

  // One 32-token chunk from a staged stage.  FULL: every token valid and copied.
  auto chunk = [&](auto full_tag, const uint8_t* st, uint32_t vaddr, int tok0, int bits) {
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
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
      const uint32_t s00 = kr0.x >> 10, s01 = kr0.y >> 10, s10 = kr1.x >> 10, s11 = kr1.y >> 10;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t mask = s <= 4 ? (0x00030003u << (2 * s)) : (0x00030003u << (2 * s - 10));
        const uint32_t a0 = (s <= 4 ? kr0.x : s00) & mask;  // row g,   channels 32t+s | 32t+8+s
        const uint32_t a1 = (s <= 4 ? kr1.x : s10) & mask;  // row g+8
        const uint32_t a2 = (s <= 4 ? kr0.y : s01) & mask;  // row g,   channels 32t+16+s | 32t+24+s
        const uint32_t a3 = (s <= 4 ? kr1.y : s11) & mask;  // row g+8
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(d[nt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
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

  bool aborted = false;
  int consumed = 0;
  for (int i = 0; i < my_chunks; ++i) {
    const int sidx = i % DEC_STAGES;
    bool ok = false;
    for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][sidx], (i / DEC_STAGES) & 1);
    ok = __all_sync(FULLM, ok);
    if (!ok) {
      if (lane == 0) flag_error(err, ERR_TIMEOUT);
      aborted = true;
      break;
    }
    consumed = i + 1;
    const uint8_t* st = stage[warp][sidx];
    const uint32_t vaddr = vrow + sidx * CHUNK;
    const int bits = sflag[warp][sidx];
    const int tok0 = (c_begin + warp + DEC_WARPS * i) * 32;
    if (tok0 + 32 <= len && bits == (int)ALL_PAGES) chunk(std::true_type{}, st, vaddr, tok0, bits);
    else chunk(std::false_type{}, st, vaddr, tok0, bits);
    __syncwarp();
    if (i + DEC_STAGES < my_chunks) issue(i + DEC_STAGES);
  }
  if (aborted) {
    // wait (bounded) for the copies still in flight before the stages go away
    for (int i = consumed; i < my_chunks && i < consumed + DEC_STAGES; ++i) {
      bool ok = false;
      for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][i % DEC_STAGES], (i / DEC_STAGES) & 1);
    }
  }
  // per-head sums over the lanes of one head (same t)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lp[nt] += __shfl_xor_sync(FULLM, lp[nt], o);
      zp[nt] += __shfl_xor_sync(FULLM, zp[nt], o);
    }
  }
  __syncthreads();  // all warps done with their stages; reuse them for the merge

  // ---- per-warp results: head 4nt+t, channels 8g + f and 64 + 8g + f ----
  float* sm_acc = reinterpret_cast<float*>(&stage[0][0][0]);  // [DEC_WARPS][G][128]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int j = 4 * nt + ti;
    if (j < G) {
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        const float sc = (float)(1 << (24 - v_pe(f)));
        sm_acc[(warp * G + j) * D + 8 * gi + f] = fmaf(fmaf(acc[nt][f][1], LO_UNSCALE, acc[nt][f][0]), sc, zp[nt]);
        sm_acc[(warp * G + j) * D + 64 + 8 * gi + f] = fmaf(fmaf(acc[nt][f][3], LO_UNSCALE, acc[nt][f][2]), sc, zp[nt]);
      }
      if (gi == 0) {
        sm_m[warp][j] = m_s[nt] * dsc[nt];
        sm_l[warp][j] = lp[nt];
      }
    }
  }
  __syncthreads();
  const int cch = threadIdx.x;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, sm_m[w][j]);
    float A = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < DEC_WARPS; ++w) {
        if (sm_m[w][j] == -INFINITY) continue;
        const float e = exp2f(sm_m[w][j] - M);
        A = fmaf(e, sm_acc[(w * G + j) * D + cch], A);
        L = fmaf(e, sm_l[w][j], L);
      }
    }
    const size_t row = ((size_t)b * n_q_heads + h * G + j) * n_splits + split;
    part.acc[row * D + cch] = A;
    if (cch == 0) {
      part.ml[row * 2] = M;
      part.ml[row * 2 + 1] = L;
    }
  }
}

// grid = (n_q_heads, n_seqs), block = 128: o = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
__global__ void __launch_bounds__(128) decode_combine_kernel(int n_q_heads, int n_splits,
                                                             Partials part, float* __restrict__ o) {
  const int j = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const size_t base = ((size_t)b * n_q_heads + j) * n_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part.ml[(base + s) * 2]);
  float A = 0.f, L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float ms = part.ml[(base + s) * 2];
      if (ms == -INFINITY) continue;
      const float e = exp2f(ms - M);
      L = fmaf(e, part.ml[(base + s) * 2 + 1], L);
      A = fmaf(e, part.acc[(base + s) * D + c], A);
    }
  }
  o[((size_t)b * n_q_heads + j) * D + c] = L > 0.f ? A / L : 0.f;
}

cudaError_t launch_decode(const PageGeom& g, int n_q_heads, int n_seqs, const void* q,
                          int q_dtype, const int32_t* seq_lens, int max_seq_len,
                          const int32_t* table, RotDev rot_k, const uint8_t* pool, int n_splits,
                          void* ws, float* o_rot, unsigned* err, cudaStream_t s) {
  (void)max_seq_len;
  if (n_seqs == 0) return cudaSuccess;
  const int gqa = n_q_heads / g.n_kv_heads;
  Partials part = partials_from_ws(ws, n_seqs, n_q_heads, n_splits);
  float* qr = rotated_q_from_ws(ws, n_seqs, n_q_heads, n_splits);
  {
    const dim3 qg(g.n_kv_heads, (n_seqs + QP_SEQS - 1) / QP_SEQS);
    if (rot_k.kind == KVQ_ROT_DENSE) {
      const size_t smem = (size_t)(D * D + QP_SEQS * gqa * D) * sizeof(float);
      static size_t attr = 0;
      if (smem > attr) {
        const cudaError_t e = cudaFuncSetAttribute(qprep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = smem;
      }
      qprep_kernel<true><<<qg, 256, smem, s>>>(n_seqs, n_q_heads, gqa, q, q_dtype, rot_k, qr);
    } else {
      qprep_kernel<false><<<qg, 256, 0, s>>>(n_seqs, n_q_heads, gqa, q, q_dtype, rot_k, qr);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  dim3 grid(n_splits, g.n_kv_heads, n_seqs);
#define KVQ_DEC(GG, PP) \
  decode_split_kernel<GG, PP><<<grid, 128, 0, s>>>(g, n_q_heads, qr, seq_lens, table, pool, n_splits, part, err)
#define KVQ_DEC_P(GG) \
  if (g.page_tokens == 16) KVQ_DEC(GG, 16); else KVQ_DEC(GG, 8)
  switch (gqa) {
    case 1: KVQ_DEC_P(1); break;
    case 2: KVQ_DEC_P(2); break;
    case 4: KVQ_DEC_P(4); break;
    case 8: KVQ_DEC_P(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_DEC_P
#undef KVQ_DEC
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(n_q_heads, n_seqs), 128, 0, s>>>(n_q_heads, n_splits, part, o_rot);
  return cudaGetLastError();
}

}  // namespace kvq
