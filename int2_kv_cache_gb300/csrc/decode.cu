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
//   sum_t p_t (z_t + s_t c_t) = sum_t (p_t s_t)(c_t - 1.5) + sum_t p_t (z_t + 1.5 s_t)
// so both contractions run on the codes c in {0,1,2,3}.
//
// Kernel structure (one CTA = one (sequence, KV head, split), 4 warps):
// * each warp owns every 4th 16-token tile of the split and streams its tiles
//   through a ring of shared-memory stages with cp.async.bulk copies completed
//   on mbarriers (one 1,152-byte page record per stage for 16-token pages, two
//   576-byte records for 8-token pages);
// * q'.c and sum_t (p_t s_t) c_t are warp-level tensor-core products
//   (mma.sync m16n8k16, fp16 inputs, fp32 accumulation).  A 2-bit field masked
//   in place inside a 16-bit word is the fp16 value c * 2^(p-24) (a subnormal,
//   p = the field's bit offset), so the operands need one logical AND per two
//   codes, and the power-of-two factor is compensated exactly in the query
//   operand.  Value codes enter as c - 1.5 (exact fp16, one OR and one packed
//   FMA per two codes) so that the running sums carry no large common term.
//   The fp32 operand of each product
//   (the rotated query, the weights p_t s_t) is split into an fp16 high part
//   and an fp16 remainder occupying the two MMA columns of one head, which
//   keeps ~22 significant bits;
// * the softmax runs online in base 2 per warp; the four warps are merged in
//   shared memory and the split's partial (m, l, unnormalised acc) is written.
// A second kernel merges the splits.
#include "quant_common.cuh"

namespace kvq {

constexpr float LOG2E = 1.4426950408889634f;
constexpr int DEC_WARPS = 4;
constexpr int DEC_STAGES = 4;
constexpr int TILE_BYTES = 1152;  // 16 tokens x 72 bytes
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

size_t decode_workspace_bytes(int n_seqs, int n_q_heads, int n_splits) {
  return (size_t)n_seqs * n_q_heads * n_splits * (D + 2) * sizeof(float);
}

int decode_auto_splits(int n_seqs, int n_kv_heads, int max_seq_len, int page_tokens) {
  (void)page_tokens;
  const int tiles = (max_seq_len + 15) / 16;
  const long long units = (long long)n_seqs * n_kv_heads;
  const int target = 152 * 4;
  int s = (int)((target + units - 1) / units);
  const int cap = tiles / 16 > 1 ? tiles / 16 : 1;  // keep >= 16 tiles per split
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
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
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

// Two 2-bit fields masked in place at bit pp (2, 4, 6 or 8) of each 16-bit half
// -> the fp16 pair (c - 1.5).  OR-ing the fp16 pattern of 1024 makes each half
// 1024 + c 2^pp exactly; one fused multiply-add by 2^-pp and -(1024 2^-pp + 1.5)
// (both exact in fp16) leaves c - 1.5 with no rounding.
__device__ __forceinline__ uint32_t centered_codes(uint32_t fields, int pp) {
  const uint32_t a = fields | 0x64006400u;
  const uint32_t sc = pp == 2 ? 0x34003400u : pp == 4 ? 0x2C002C00u : pp == 6 ? 0x24002400u : 0x1C001C00u;
  const uint32_t bi = pp == 2 ? 0xDC06DC06u : pp == 4 ? 0xD418D418u : pp == 6 ? 0xCC60CC60u : 0xC580C580u;
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(sc), "r"(bi));
  return d;
}

// Byte offsets of token row r (0..15) inside a staged tile.
template <int P>
struct TileLayout {
  static __device__ __forceinline__ int k(int r) { return P == 16 ? 32 * r : (r >> 3) * 576 + 32 * (r & 7); }
  static __device__ __forceinline__ int v(int r) { return P == 16 ? 512 + 32 * r : (r >> 3) * 576 + 256 + 32 * (r & 7); }
  static __device__ __forceinline__ int km(int r) { return P == 16 ? 1024 + 4 * r : (r >> 3) * 576 + 512 + 4 * (r & 7); }
  static __device__ __forceinline__ int vm(int r) { return P == 16 ? 1088 + 4 * r : (r >> 3) * 576 + 544 + 4 * (r & 7); }
};

__device__ __forceinline__ float2 meta_pair(const uint8_t* p) {
  const uint32_t m = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(__half2float(__ushort_as_half((unsigned short)(m & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(m >> 16))));
}

// ---------------------------------------------------------------------------
// The split kernel.  grid = (n_splits, n_kv_heads, n_seqs), block = 128.
// G = query heads per KV head; NT = n-tiles of 8 columns (2 columns per head).
// ---------------------------------------------------------------------------
template <int G, int P>
__global__ void __launch_bounds__(128) decode_split_kernel(
    PageGeom g, int n_q_heads, const void* __restrict__ q, int q_dtype,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ table, RotDev rot_k,
    const uint8_t* __restrict__ pool, int n_splits, Partials part, unsigned* err) {
  constexpr int NT = (G + 3) / 4;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;  // MMA group id, thread id in group

  __shared__ __align__(128) uint8_t stage[DEC_WARPS][DEC_STAGES][TILE_BYTES];
  __shared__ __align__(8) uint64_t bars[DEC_WARPS][DEC_STAGES];
  __shared__ __align__(16) float qs[G][D];
  __shared__ float qsum[G], qexp[G];
  __shared__ float sm_m[DEC_WARPS][G], sm_l[DEC_WARPS][G];
  __shared__ uint8_t sflag[DEC_WARPS][DEC_STAGES];  // bit 0 / bit 1: first / second page copied

  int len = __ldg(seq_lens + b);
  if (len < 0 || len > g.max_blocks * g.page_tokens) {
    if (threadIdx.x == 0) flag_error(err, ERR_SEQ_RANGE);
    len = 0;
  }
  const int n_pages = (len + P - 1) / P;
  const int n_tiles = (len + 15) / 16;
  const int tps = (n_tiles + n_splits - 1) / n_splits;
  const int t_begin = split * tps;
  const int t_end = min(n_tiles, t_begin + tps);
  const int my_tiles = t_end > t_begin + warp ? (t_end - t_begin - warp + DEC_WARPS - 1) / DEC_WARPS : 0;
  const int32_t* trow = table + (size_t)b * g.max_blocks;

  // Page ids of the warp's tiles, 32 tiles at a time in lane registers (lane l
  // holds tile i0 + l); the producer reads them with shuffles.
  int pc0 = -1, pc1 = -1;
  auto fill_cache = [&](int i0) {
    const int i = i0 + lane;
    const int tile = t_begin + warp + DEC_WARPS * i;
    pc0 = -1;
    pc1 = -1;
    if (i < my_tiles) {
      if (P == 16) {
        pc0 = __ldg(trow + tile);
      } else {
        pc0 = __ldg(trow + 2 * tile);
        pc1 = 2 * tile + 1 < n_pages ? __ldg(trow + 2 * tile + 1) : -2;  // -2: no second page
      }
    }
  };
  // Issue the copy of the warp's i-th tile into its stage.  Called by the whole warp.
  auto issue = [&](int i) {
    if (i % 32 == 0 && i > 0) fill_cache(i);
    const int blk0 = __shfl_sync(0xffffffffu, pc0, i % 32);
    const int blk1 = __shfl_sync(0xffffffffu, pc1, i % 32);
    if (lane == 0) {
      const int sidx = i % DEC_STAGES;
      uint64_t* bar = &bars[warp][sidx];
      uint8_t* dst = stage[warp][sidx];
      const bool ok0 = blk0 >= 0 && blk0 < g.num_blocks;
      const bool ok1 = P == 16 ? ok0 : (blk1 >= 0 && blk1 < g.num_blocks);
      if (!ok0 || (P == 8 && blk1 != -2 && !ok1)) flag_error(err, ERR_BLOCK_RANGE);
      sflag[warp][sidx] = (ok0 ? 1 : 0) | (ok1 ? 2 : 0);
      fence_proxy_async();
      const size_t stride = (size_t)g.n_kv_heads * g.record;
      const uint8_t* base = pool + (size_t)h * g.record;
      if (P == 16) {
        if (ok0) {
          mbar_arrive_expect_tx(bar, TILE_BYTES);
          bulk_g2s(dst, base + (size_t)blk0 * stride, TILE_BYTES, bar);
        } else {
          mbar_arrive(bar);
        }
      } else {
        const uint32_t bytes = (ok0 ? 576u : 0u) + (ok1 ? 576u : 0u);
        if (bytes) {
          mbar_arrive_expect_tx(bar, bytes);
          if (ok0) bulk_g2s(dst, base + (size_t)blk0 * stride, 576, bar);
          if (ok1) bulk_g2s(dst + 576, base + (size_t)blk1 * stride, 576, bar);
        } else {
          mbar_arrive(bar);
        }
      }
    }
  };

  if (lane == 0) {
    for (int s = 0; s < DEC_STAGES; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  fill_cache(0);
  for (int i = 0; i < DEC_STAGES && i < my_tiles; ++i) issue(i);

  // ---- prologue: q'_j = q_j R_K,h * log2(e)/sqrt(128) (Eq. 22) ----
  for (int jj = warp; jj < G; jj += DEC_WARPS) {
    float4 v = load4(q, ((size_t)b * n_q_heads + h * G + jj) * D + 4 * lane, q_dtype);
    v = rotate_vec_warp(v, rot_k, h, lane, false);
    const float sc = LOG2E * INV_SQRT_D;
    v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
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
  // fp16 high part of q'_j * 2^(8-pe-e_j), column 2j+1 the remainder.
  uint32_t bq[NT][8][2];
  {
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
  }
  float my_qsum[NT], my_dscale[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int j = 4 * nt + ti;
    my_qsum[nt] = j < G ? qsum[j] : 0.f;
    my_dscale[nt] = j < G ? exp2f(16.f + qexp[j]) : 0.f;
  }

  float m[NT], l[NT], zacc[NT];
  float acc[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt] = -INFINITY;
    l[nt] = 0.f;
    zacc[nt] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[nt][i][0] = acc[nt][i][1] = acc[nt][i][2] = acc[nt][i][3] = 0.f;
  }

  bool aborted = false;
  int consumed = 0;
  for (int i = 0; i < my_tiles; ++i) {
    const int tile = t_begin + warp + DEC_WARPS * i;
    const int sidx = i % DEC_STAGES;
    bool ok = false;
    for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][sidx], (i / DEC_STAGES) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0) flag_error(err, ERR_TIMEOUT);
      aborted = true;
      break;
    }
    consumed = i + 1;
    const uint8_t* st = stage[warp][sidx];
    // rows valid: position < len and its page's block id in range
    const int nv = min(16, len - tile * 16);
    const int fl = sflag[warp][sidx];
    const bool half_ok[2] = {(fl & 1) != 0, (fl & 2) != 0};
    const bool row0_ok = gi < nv && half_ok[0];
    const bool row1_ok = gi + 8 < nv && half_ok[1];

    // ---- scores: D[token][2j + {hi,lo}] = 2^-16 * sum_c code * q'_j[c] ----
    const uint2 kr0 = *reinterpret_cast<const uint2*>(st + TileLayout<P>::k(gi) + 8 * ti);
    const uint2 kr1 = *reinterpret_cast<const uint2*>(st + TileLayout<P>::k(gi + 8) + 8 * ti);
    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
    {
      const uint32_t k00 = kr0.x, k01 = kr0.y, k10 = kr1.x, k11 = kr1.y;
      const uint32_t s00 = k00 >> 10, s01 = k01 >> 10, s10 = k10 >> 10, s11 = k11 >> 10;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t mask = s <= 4 ? (0x00030003u << (2 * s)) : (0x00030003u << (2 * s - 10));
        const uint32_t a0 = (s <= 4 ? k00 : s00) & mask;  // row g,   channels 32t+s | 32t+8+s
        const uint32_t a1 = (s <= 4 ? k10 : s10) & mask;  // row g+8
        const uint32_t a2 = (s <= 4 ? k01 : s01) & mask;  // row g,   channels 32t+16+s | 32t+24+s
        const uint32_t a3 = (s <= 4 ? k11 : s11) & mask;  // row g+8
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(d[nt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
      }
    }
    const float2 km0 = meta_pair(st + TileLayout<P>::km(gi));
    const float2 km1 = meta_pair(st + TileLayout<P>::km(gi + 8));
    const float2 vm0 = meta_pair(st + TileLayout<P>::vm(gi));
    const float2 vm1 = meta_pair(st + TileLayout<P>::vm(gi + 8));

    uint32_t bp[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float dot0 = fmaf(d[nt][1], LO_UNSCALE, d[nt][0]) * my_dscale[nt];
      const float dot1 = fmaf(d[nt][3], LO_UNSCALE, d[nt][2]) * my_dscale[nt];
      const float sc0 = row0_ok ? fmaf(km0.x, dot0, km0.y * my_qsum[nt]) : -INFINITY;
      const float sc1 = row1_ok ? fmaf(km1.x, dot1, km1.y * my_qsum[nt]) : -INFINITY;
      float mx = fmaxf(sc0, sc1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const bool need = mx > m[nt] + TAU;  // reference max moves only by > TAU
      const float alpha = need ? exp2f(m[nt] - mx) : 1.f;
      if (need) m[nt] = mx;
      const float msafe = m[nt] == -INFINITY ? 0.f : m[nt];
      const float p0 = exp2f(sc0 - msafe), p1 = exp2f(sc1 - msafe);
      float ps = p0 + p1;
      float pz = (row0_ok ? p0 * fmaf(1.5f, vm0.x, vm0.y) : 0.f) + (row1_ok ? p1 * fmaf(1.5f, vm1.x, vm1.y) : 0.f);
      ps += __shfl_xor_sync(0xffffffffu, ps, 4);
      pz += __shfl_xor_sync(0xffffffffu, pz, 4);
      ps += __shfl_xor_sync(0xffffffffu, ps, 8);
      pz += __shfl_xor_sync(0xffffffffu, pz, 8);
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);
      pz += __shfl_xor_sync(0xffffffffu, pz, 16);
      l[nt] = fmaf(l[nt], alpha, ps);
      zacc[nt] = fmaf(zacc[nt], alpha, pz);
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          acc[nt][r][0] *= alpha; acc[nt][r][1] *= alpha; acc[nt][r][2] *= alpha; acc[nt][r][3] *= alpha;
        }
      }
      // weights p_t s_t of this lane's rows, then gathered into the B fragment:
      // k = 2t, 2t+1, 2t+8, 2t+9 <-> tokens t, t+4, t+8, t+12; column g <-> head g/2, part g&1
      const float w0 = row0_ok ? p0 * vm0.x : 0.f;
      const float w1 = row1_ok ? p1 * vm1.x : 0.f;
      const int src_a = ti * 4 + (gi >> 1), src_b = (ti + 4) * 4 + (gi >> 1);
      const float x0 = __shfl_sync(0xffffffffu, w0, src_a);
      const float x1 = __shfl_sync(0xffffffffu, w0, src_b);
      const float x2 = __shfl_sync(0xffffffffu, w1, src_a);
      const float x3 = __shfl_sync(0xffffffffu, w1, src_b);
      if (gi & 1) {
        bp[nt][0] = pack_half2((x0 - half_rn(x0)) * LO_SCALE, (x1 - half_rn(x1)) * LO_SCALE);
        bp[nt][1] = pack_half2((x2 - half_rn(x2)) * LO_SCALE, (x3 - half_rn(x3)) * LO_SCALE);
      } else {
        bp[nt][0] = pack_half2(x0, x1);
        bp[nt][1] = pack_half2(x2, x3);
      }
    }

    // ---- values: D[channel][2j + {hi,lo}] += sum_t (code - 1.5) * p_t s_t ----
    // Zero-mean codes keep the running sums free of the large common term
    // 1.5 sum_t p_t s_t (which is carried, exactly cancelled, in the zero term).
    {
      const uint32_t wa = *reinterpret_cast<const uint32_t*>(st + TileLayout<P>::v(ti) + 4 * gi);
      const uint32_t wb = *reinterpret_cast<const uint32_t*>(st + TileLayout<P>::v(ti + 4) + 4 * gi);
      const uint32_t wc = *reinterpret_cast<const uint32_t*>(st + TileLayout<P>::v(ti + 8) + 4 * gi);
      const uint32_t wd = *reinterpret_cast<const uint32_t*>(st + TileLayout<P>::v(ti + 12) + 4 * gi);
      const uint32_t w[4] = {prmt(wa, wb, 0x5410), prmt(wa, wb, 0x7632),   // channels 16g+0..7 | 16g+8..15,
                             prmt(wc, wd, 0x5410), prmt(wc, wd, 0x7632)};  // tokens t|t+4, then t+8|t+12
      uint32_t wl[4], wr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wl[u] = w[u] << 2;
        wr[u] = w[u] >> 8;
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        // field of channel 16g + r (or 16g + 8 + r) at bit pp of each half after the shift
        const int pp = r == 0 ? 2 : (r <= 4 ? 2 * r : 2 * r - 8);
        const uint32_t mask = 0x00030003u << pp;
        uint32_t a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t src = r == 0 ? wl[u] : (r <= 4 ? w[u] : wr[u]);
          a[u] = centered_codes(src & mask, pp);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt][r], a[0], a[1], a[2], a[3], bp[nt][0], bp[nt][1]);
      }
    }
    __syncwarp();
    if (i + DEC_STAGES < my_tiles) issue(i + DEC_STAGES);
  }
  if (aborted) {
    // wait (bounded) for the copies still in flight before the stages go away
    for (int i = consumed; i < my_tiles && i < consumed + DEC_STAGES; ++i) {
      bool ok = false;
      for (int it = 0; it < WAIT_LIMIT && !ok; ++it) ok = mbar_try_wait(&bars[warp][i % DEC_STAGES], (i / DEC_STAGES) & 1);
    }
  }
  __syncthreads();  // all warps done with their stages; reuse them for the merge

  // ---- per-warp results: head 4nt+t, channels 16g + r and 16g + 8 + r ----
  float* sm_acc = reinterpret_cast<float*>(&stage[0][0][0]);  // [DEC_WARPS][G][128]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int j = 4 * nt + ti;
    if (j < G) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        sm_acc[(warp * G + j) * D + 16 * gi + r] = fmaf(acc[nt][r][1], LO_UNSCALE, acc[nt][r][0]) + zacc[nt];
        sm_acc[(warp * G + j) * D + 16 * gi + 8 + r] = fmaf(acc[nt][r][3], LO_UNSCALE, acc[nt][r][2]) + zacc[nt];
      }
      if (gi == 0) {
        sm_m[warp][j] = m[nt];
        sm_l[warp][j] = l[nt];
      }
    }
  }
  __syncthreads();
  const int c = threadIdx.x;
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
        A = fmaf(e, sm_acc[(w * G + j) * D + c], A);
        L = fmaf(e, sm_l[w][j], L);
      }
    }
    const size_t row = ((size_t)b * n_q_heads + h * G + j) * n_splits + split;
    part.acc[row * D + c] = A;
    if (c == 0) {
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
  dim3 grid(n_splits, g.n_kv_heads, n_seqs);
#define KVQ_DEC(GG, PP) \
  decode_split_kernel<GG, PP><<<grid, 128, 0, s>>>(g, n_q_heads, q, q_dtype, seq_lens, table, rot_k, pool, n_splits, part, err)
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
