// Bulk cache write for dense rotations on the fifth-generation tensor cores.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization", §6 (the cache-write
// kernel: rotate, subtract mu R, clip, quantize, pack and write in one launch)
// with a dense learned R = R0 exp(A - A^T) (§4.2 Eq. 11), the rotation being a
// [tokens x 128] x [128 x 128] product per KV head.  The group quantizer and its
// exact decisions are those of quant_common.cuh (Eq. 4, group 128, fp16 scale
// and zero).
//
// Arithmetic.  Every fp32 R with |R| >= 2^-100 splits exactly into three bf16 limbs,
//   R = hi + mid + lo, hi = bf16(R), mid = bf16(R - hi), lo = R - hi - mid
// (round to nearest: |mid| <= 2^-8 |R|, and R - hi - mid has at most 8
// significant bits, so lo holds it exactly; (lo + mid) + hi gives R back in fp32
// without rounding); smaller values are split with an error of at most 2^-134.  fp32
// inputs x split the same way; bf16 inputs are one limb.
// The tensor cores take bf16 x bf16 products (exact in fp32) into fp32
// accumulators in tensor memory.  Their accumulation order and rounding are not
// documented, so the error bound charges every 128 x 128 x 16 MMA
//   96 u (|D| + sum |a_j b_j|)       (u = 2^-24)
// for its accumulator D: the worst case of adding the 16 exact products to D in
// any chunking, every chunk aligned to its largest addend and truncated to fp32
// precision, then rounded or truncated again.  To keep |D| small, accumulator a
// (of four, 128 columns each: all of tensor memory) takes only K steps 2a and
// 2a + 1, limbs in the order lo, mid, hi, so that its error is at most
// 96 u (2 P_0 + P_1 + small terms) <= 195 u P_a, with P_k = sum over the
// channels c of step k of |x_c| |R_cd|.  Over the four accumulators, their fp32
// sum, and (fp32 input) the three dropped limb products of order 2^-24, the
// rotated value is within 210 u sum_c |x_c| |R_cd| <= 210 u ||x|| ||R_:,d|| of
// x R (Cauchy-Schwarz), plus 1e-30 for products that could be flushed as
// subnormals and for the split of values below 2^-100.
//
// Decisions.  One thread owns a quarter of one token's group: an accumulator row
// and 32 of its columns (the four warps of a tensor-memory lane quarter share a
// row and meet at named barriers to combine the row's extremes).  Scale and zero
// are taken from the fp32 min and max when certain under that bound
// (qparams_certain), codes by the scaled distance of (y - z) / s to the nearest
// half-integer.  Where a decision is uncertain, the elements that can decide it
// (for scale and zero: the columns within 2E of the fp32 extremes, which hold the
// exact arg-min and arg-max) are evaluated again by the whole warp from the staged
// bf16 limbs of x and R (lane l takes channels 4l..4l+3): first in fp32 (an FMA
// chain and a shuffle tree, 9 u sum_c |x_c R_cd|), then, where still uncertain, in
// double-float (exact products by FMA, compensated sums), deciding with
// qparams_df / qcode_df.  An uncertain element costs about 50 (fp32) or 150
// (double-float) warp instructions instead of a whole group's double-float
// rotation.  The result equals the decision on the exact x R - mu R except within
// ~1e-12 (relative) of a rounding boundary, like the double-float path elsewhere.
//
// Schedule.  One CTA per SM (tensor memory: 512 columns), persistent over units
// (role, KV head, 128-token tile), ordered so that consecutive units share R_h:
//   stage R_h's limbs (B operand, [d][c], 128-byte swizzle) when the head changes;
//   the tile's x (A operand, [token][c]): bf16 by asynchronous copies one unit
//   ahead into a second buffer, fp32 loaded and split here; the tokens' pages located;
//   one thread issues the 24 (bf16) or 48 (fp32) MMAs and commits them to an
//   mbarrier; all threads wait (bounded) and read the accumulators, after which the
//   next unit's MMAs are issued (same head) while this unit's decisions are taken.
// grid = min(units, SMs), block = 512.
#include <algorithm>

#include "quant_common.cuh"
#include "tcgen05.cuh"

namespace kvq {

constexpr int ATC_M = 128;                 // tokens per tile (accumulator rows)
constexpr int ATC_THREADS = 512;
constexpr int ATC_PARTS = 4;               // column parts of a row (one warp each per lane quarter)
constexpr int ATC_TILE = 128 * 128 * 2;    // one bf16 operand tile [128 rows][128 K] (two 64-wide K halves)
constexpr int ATC_HALF = 128 * 128;        // one K half: 128 rows of 128 bytes
constexpr float ATC_EREL = 1.2517e-05f;    // 210 u
constexpr float ATC_EABS = 1e-30f;

__host__ __device__ constexpr int atc_smem_bytes(bool f32) { return 1024 + (3 + (f32 ? 3 : 2)) * ATC_TILE; }

// Byte offset of element (row r, K index k) in an operand tile: K half k / 64,
// rows of 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t atc_off(int r, int k) {
  return (uint32_t)((k >> 6) * ATC_HALF + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1));
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_val(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Exact three-limb split of eight fp32 values into bf16 hi / mid / lo chunks.
__device__ __forceinline__ void split3_8(const float (&v)[8], uint4& h, uint4& m, uint4& l) {
  uint32_t hw[4], mw[4], lw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t hb[2], mb[2], lb[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float x = v[2 * i + j];
      hb[j] = bf16_bits_rn(x);
      const float r1 = __fsub_rn(x, bf16_val(hb[j]));
      mb[j] = bf16_bits_rn(r1);
      lb[j] = bf16_bits_rn(__fsub_rn(r1, bf16_val(mb[j])));  // exact
    }
    hw[i] = hb[0] | (hb[1] << 16);
    mw[i] = mb[0] | (mb[1] << 16);
    lw[i] = lb[0] | (lb[1] << 16);
  }
  h = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  m = make_uint4(mw[0], mw[1], mw[2], mw[3]);
  l = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// Four consecutive bf16 values (8 bytes at a 8-byte aligned shared address) as floats.
__device__ __forceinline__ void lds_bf4(const uint8_t* p, float (&f)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xffff0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xffff0000u);
}

// Double-float value of (x_m R)_d - mu for row m of the staged x and column d of
// the staged R; every lane of the warp takes part and returns the total.
template <bool F32>
__device__ __forceinline__ DF atc_df_item(const uint8_t* sA, const uint8_t* sB, int m, int d, float mu, int lane) {
  const int k = 4 * lane;
  const uint32_t oa = atc_off(m, k), ob = atc_off(d, k);
  float x[4], rh[4], rm[4], rl[4];
  lds_bf4(sA + oa, x);
  if (F32) {
    float xm[4], xl[4];
    lds_bf4(sA + ATC_TILE + oa, xm);
    lds_bf4(sA + 2 * ATC_TILE + oa, xl);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __fadd_rn(__fadd_rn(xl[i], xm[i]), x[i]);  // exact
  }
  lds_bf4(sB + ob, rh);
  lds_bf4(sB + ATC_TILE + ob, rm);
  lds_bf4(sB + 2 * ATC_TILE + ob, rl);
  float sh = 0.f, sl = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float r = __fadd_rn(__fadd_rn(rl[i], rm[i]), rh[i]);  // R exactly
    const float p = __fmul_rn(x[i], r);
    const float e = __fmaf_rn(x[i], r, -p);  // x r = p + e exactly
    const DF t = two_sum(sh, p);
    sh = t.hi;
    sl = __fadd_rn(sl, __fadd_rn(t.lo, e));
  }
  DF acc = df_norm(sh, sl);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = df_add(acc, shfl_xor_df(acc, o));
  return df_add_f(acc, -mu);
}

// One round of warp-wide double-float evaluations: every lane with a pending
// column (the lowest set bit of `pending`, in this lane's row row0 + lane) has it
// evaluated by the whole warp and cleared; returns that column (-1 if none) and
// its value in `v`.  Callers repeat rounds while any lane has pending columns.
template <bool F32>
__device__ __forceinline__ int atc_round(uint32_t& pending, const uint8_t* sA, const uint8_t* sB, const float* s_mu,
                                         int row0, int col0, int lane, DF& v) {
  constexpr unsigned FULLM = 0xffffffffu;
  const int my_d = pending ? __ffs(pending) - 1 : -1;
  if (pending) pending &= pending - 1u;
  unsigned act = __ballot_sync(FULLM, my_d >= 0);
  v = DF{0.f, 0.f};
  while (act) {
    const int src = __ffs(act) - 1;
    act &= act - 1u;
    const int d = __shfl_sync(FULLM, my_d, src);
    const DF t = atc_df_item<F32>(sA, sB, row0 + src, col0 + d, s_mu[col0 + d], lane);
    if (lane == src) v = t;
  }
  return my_d;
}

// fp32 value of (x_m R)_d - mu with the same staged operands (the middle tier):
// lane l forms channels 4l..4l+3 by an FMA chain, then a 5-level shuffle tree.
// Off by at most 9 u sum_c |x_c R_cd| (4 + 5 roundings) + u (|v| + |mu|).
template <bool F32>
__device__ __forceinline__ float atc_f32_item(const uint8_t* sA, const uint8_t* sB, int m, int d, float mu, int lane) {
  const int k = 4 * lane;
  const uint32_t oa = atc_off(m, k), ob = atc_off(d, k);
  float x[4], rh[4], rm[4], rl[4];
  lds_bf4(sA + oa, x);
  if (F32) {
    float xm[4], xl[4];
    lds_bf4(sA + ATC_TILE + oa, xm);
    lds_bf4(sA + 2 * ATC_TILE + oa, xl);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __fadd_rn(__fadd_rn(xl[i], xm[i]), x[i]);
  }
  lds_bf4(sB + ob, rh);
  lds_bf4(sB + ATC_TILE + ob, rm);
  lds_bf4(sB + 2 * ATC_TILE + ob, rl);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) s = __fmaf_rn(x[i], __fadd_rn(__fadd_rn(rl[i], rm[i]), rh[i]), s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return __fsub_rn(s, mu);
}

// One round of the middle tier: as atc_round, with fp32 values.
template <bool F32>
__device__ __forceinline__ int atc_round_f32(uint32_t& pending, const uint8_t* sA, const uint8_t* sB,
                                             const float* s_mu, int row0, int col0, int lane, float& v) {
  constexpr unsigned FULLM = 0xffffffffu;
  const int my_d = pending ? __ffs(pending) - 1 : -1;
  if (pending) pending &= pending - 1u;
  unsigned act = __ballot_sync(FULLM, my_d >= 0);
  v = 0.f;
  while (act) {
    const int src = __ffs(act) - 1;
    act &= act - 1u;
    const int d = __shfl_sync(FULLM, my_d, src);
    const float t = atc_f32_item<F32>(sA, sB, row0 + src, col0 + d, s_mu[col0 + d], lane);
    if (lane == src) v = t;
  }
  return my_d;
}

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void set_code(uint32_t (&packed)[2], int d, unsigned c) {
  const int sh = 2 * (d & 15);
  if (d < 16) packed[0] = (packed[0] & ~(3u << sh)) | (c << sh);
  else packed[1] = (packed[1] & ~(3u << sh)) | (c << sh);
}

template <bool F32>
__global__ void __launch_bounds__(ATC_THREADS, 1) append_dense_tc_kernel(
    PageGeom g, int n_seqs, int n_new, const int32_t* __restrict__ cu_new,
    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ table, AppendRoles roles, int n_roles,
    uint8_t* __restrict__ pool, unsigned* err) {
  constexpr unsigned FULLM = 0xffffffffu;
  constexpr uint32_t IDESC = idesc_bf16_f32(ATC_M, 128);
  extern __shared__ uint8_t atc_raw[];
  uint8_t* sB = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(atc_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA0 = sB + 3 * ATC_TILE;  // fp32 x: three limb tiles; bf16 x: two buffers of one tile
  __shared__ float s_mu[128];      // mu R_h (keys with centring), else 0
  __shared__ float s_nrm[ATC_M];   // upper bound of ||x|| per row
  __shared__ long long s_rec[ATC_M];
  __shared__ int s_slot[ATC_M];
  __shared__ float s_ex[2][ATC_PARTS][2][ATC_M];  // [tier][column part][min, max] per row
  __shared__ float2 s_dex[ATC_PARTS][2][ATC_M];   // double-float [column part][min, max] per row
  __shared__ float s_red[2][8];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = g.n_kv_heads;
  const int tiles = (n_new + ATC_M - 1) / ATC_M;
  const long long units = (long long)n_roles * H * tiles;
  const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // loader role: row r of the tile, channels 32 kq .. 32 kq + 31; epilogue role:
  // accumulator row m (lane quarter q4) and columns 32 cp .. 32 cp + 31
  const int r = tid >> 2, kq = tid & 3;
  const int q4 = warp & 3, cp = warp >> 2, m = 32 * q4 + lane;
  auto unit_of = [&](long long u, int& rh, int& tile, int& h, AppendRole& ro) {
    rh = (int)(u / tiles);
    tile = (int)(u % tiles);
    h = rh % H;
    ro = rh / H ? roles.r[1] : roles.r[0];
  };
  auto buf = [&](long long u) { return F32 ? sA0 : sA0 + (int)((u - u0) & 1) * ATC_TILE; };
  // bf16 x: asynchronous copies of a unit's rows into its buffer (zero rows past the end)
  auto prefetch = [&](long long u) {
    if (F32 || u >= u1) return;
    int rh, tile, h;
    AppendRole ro;
    unit_of(u, rh, tile, h, ro);
    const int t = tile * ATC_M + r;
    const bool in = t < n_new;
    const __nv_bfloat16* src =
        static_cast<const __nv_bfloat16*>(ro.src) + ((size_t)(in ? t : 0) * H + h) * D + 32 * kq;
    uint8_t* dst = buf(u);
#pragma unroll
    for (int j = 0; j < 4; ++j) cp_async16_zfill(dst + atc_off(r, 32 * kq + 8 * j), src + 8 * j, in ? 16u : 0u);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // a unit's A operand (fp32 x: loaded and split here; bf16 x: its copies have landed),
  // row norms and token pages; ends with the proxy fence for the tensor cores
  auto prepare = [&](long long u) {
    int rh, tile, h;
    AppendRole ro;
    unit_of(u, rh, tile, h, ro);
    const int t0 = tile * ATC_M, t = t0 + r;
    uint8_t* sA = buf(u);
    float ss = 0.f;
    if (F32) {
      const float4* src =
          reinterpret_cast<const float4*>(static_cast<const float*>(ro.src) + ((size_t)t * H + h) * D + 32 * kq);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), b4 = a4;
        if (t < n_new) {
          a4 = __ldg(src + 2 * j);
          b4 = __ldg(src + 2 * j + 1);
        }
        const float v[8] = {a4.x, a4.y, a4.z, a4.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
        uint4 lh, lm, ll;
        split3_8(v, lh, lm, ll);
        const uint32_t o = atc_off(r, 32 * kq + 8 * j);
        *reinterpret_cast<uint4*>(sA + o) = lh;
        *reinterpret_cast<uint4*>(sA + ATC_TILE + o) = lm;
        *reinterpret_cast<uint4*>(sA + 2 * ATC_TILE + o) = ll;
      }
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's copies of the unit
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(sA + atc_off(r, 32 * kq + 8 * j));
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __uint_as_float(q[i] << 16), hi = __uint_as_float(q[i] & 0xffff0000u);
          ss = fmaf(lo, lo, ss);
          ss = fmaf(hi, hi, ss);
        }
      }
    }
    ss += __shfl_xor_sync(FULLM, ss, 1);
    ss += __shfl_xor_sync(FULLM, ss, 2);
    if (kq == 0) s_nrm[r] = sqrtf(ss) * 1.0001f;
    if (tid < ATC_M) {
      long long rec = -1;
      int slot = 0;
      if (t0 + tid < n_new && !locate(t0 + tid, n_seqs, cu_new, start_pos, table, g, err, &rec, &slot, 0)) rec = -1;
      s_rec[tid] = rec < 0 ? -1 : rec + h;
      s_slot[tid] = slot;
    }
    fence_proxy_async();  // the tensor cores read A through the async proxy
  };
  auto issue = [&](long long u) {  // thread 0: the unit's 128 x 128 x 128 product into four accumulators
    tc_fence_after();
    const uint64_t a0 = sw128_desc(buf(u)), b0 = sw128_desc(sB);
    const uint64_t tile_step = ATC_TILE >> 4, half_step = ATC_HALF >> 4;  // descriptor address units
    auto desc = [&](uint64_t base, int limb, int ks) {
      return base + (uint64_t)limb * tile_step + (uint64_t)(ks >> 2) * half_step + 2 * (ks & 3);
    };
    // (x limb, R limb) pairs from the smallest products to the largest (limb 0 = hi):
    // fp32 x: (lo, hi) (mid, mid) (hi, lo), then (mid, hi) (hi, mid), then (hi, hi);
    // bf16 x: (x, lo), (x, mid), (x, hi)
    constexpr int NP = F32 ? 6 : 3;
    constexpr uint32_t PX = F32 ? 0x001012u : 0u;      // x limb of pair p: bits 4p .. 4p + 3
    constexpr uint32_t PR = F32 ? 0x010210u : 0x012u;  // R limb of pair p
#pragma unroll
    for (int a = 0; a < 4; ++a) {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int ks = 2 * a + s;
          tc_mma_bf16(tmem + 128 * a, desc(a0, (PX >> (4 * p)) & 15, ks), desc(b0, (PR >> (4 * p)) & 15, ks), IDESC,
                      p > 0 || s > 0);
        }
      }
    }
    tc_commit(&s_bar);
  };
  prefetch(u0);
  if (u0 < u1) prepare(u0);
  prefetch(u0 + 1);
  int cur = -1;
  float cn_max = 0.f, mu_max = 0.f;
  uint32_t phase = 0;
  bool alive = true, issued = false;
  for (long long u = u0; u < u1 && alive; ++u) {
    int rh, tile, h;
    AppendRole ro;
    unit_of(u, rh, tile, h, ro);
    const uint8_t* sA = buf(u);
    if (rh != cur) {
      // ---- stage R_h as three limb tiles: row d, K = c holds limb j of R[c][d] ----
      __syncthreads();  // the previous unit's items have read the old limbs
      const float* R = ro.rot.dense + (size_t)h * D * D;
      const int d = tid & 127;
      float ss = 0.f;
      for (int ch = tid >> 7; ch < 16; ch += ATC_THREADS / 128) {  // channels 8 ch .. 8 ch + 7
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[i] = __ldg(R + (size_t)(8 * ch + i) * D + d);  // a warp reads 128 contiguous bytes per i
          ss = fmaf(v[i], v[i], ss);
        }
        uint4 lh, lm, ll;
        split3_8(v, lh, lm, ll);
        const uint32_t o = atc_off(d, 8 * ch);
        *reinterpret_cast<uint4*>(sB + o) = lh;
        *reinterpret_cast<uint4*>(sB + ATC_TILE + o) = lm;
        *reinterpret_cast<uint4*>(sB + 2 * ATC_TILE + o) = ll;
      }
      fence_proxy_async();
      float* s_ss = &s_ex[0][0][0][0];  // column sums of squares over the channel parts
      s_ss[tid] = ss;
      if (tid < 128) s_mu[tid] = ro.mu_rot ? __ldg(ro.mu_rot + (size_t)h * D + tid) : 0.f;
      __syncthreads();
      if (tid < 128) {
        float cs = 0.f;
#pragma unroll
        for (int i = 0; i < ATC_THREADS / 128; ++i) cs += s_ss[tid + 128 * i];
        const float cn = warp_max(sqrtf(cs));
        const float mm = warp_max(fabsf(s_mu[tid]));
        if (lane == 0) {
          s_red[0][warp] = cn;
          s_red[1][warp] = mm;
        }
      }
      __syncthreads();
      cn_max = fmaxf(fmaxf(s_red[0][0], s_red[0][1]), fmaxf(s_red[0][2], s_red[0][3])) * 1.0001f;
      mu_max = fmaxf(fmaxf(s_red[1][0], s_red[1][1]), fmaxf(s_red[1][2], s_red[1][3]));
      cur = rh;
    }
    if (!issued) {
      __syncthreads();  // the operands of u are staged and fenced
      if (tid == 0) issue(u);
      __syncwarp();
    }
    bool ok = mbar_wait_bounded(&s_bar, phase);
    phase ^= 1u;
    if (!__syncthreads_and(ok)) {
      if (tid == 0) flag_error(err, ERR_TIMEOUT);
      alive = false;
      break;
    }
    tc_fence_after();
    // ---- accumulators -> y (this thread: row m, columns 32 cp .. 32 cp + 31) ----
    float y[32];
    {
      const uint32_t tb = tmem + ((uint32_t)(32 * q4) << 16) + 32 * cp;
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float s0[8], s1[8];
        tmem_ld8(tb + 8 * c8, s0);
#pragma unroll
        for (int a = 1; a < 4; ++a) {
          tmem_ld8(tb + 128 * a + 8 * c8, s1);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float2 t = f2up(f2add(f2pk(s0[i], s0[i + 1]), f2pk(s1[i], s1[i + 1])));
            s0[i] = t.x;
            s0[i + 1] = t.y;
          }
        }
        const float4 mu0 = *reinterpret_cast<const float4*>(s_mu + 32 * cp + 8 * c8);
        const float4 mu1 = *reinterpret_cast<const float4*>(s_mu + 32 * cp + 8 * c8 + 4);
        const float mus[8] = {mu0.x, mu0.y, mu0.z, mu0.w, mu1.x, mu1.y, mu1.z, mu1.w};
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 t = f2up(f2sub(f2pk(s0[i], s0[i + 1]), f2pk(mus[i], mus[i + 1])));
          y[8 * c8 + i] = t.x;
          y[8 * c8 + i + 1] = t.y;
        }
      }
    }
    // the next unit's copies have landed: its product may start once tensor memory is read
    if (!F32) asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    bool early = false;
    if (!F32 && u + 1 < u1) {
      int rh1, tile1, h1;
      AppendRole ro1;
      unit_of(u + 1, rh1, tile1, h1, ro1);
      early = rh1 == rh;
    }
    if (early && tid == 0) issue(u + 1);
    const bool valid = s_rec[m] >= 0;
    const float bnd = s_nrm[m] * cn_max;  // >= sum_c |x_c R_cd| for every column d
    float E = __fmaf_rn(ATC_EREL, bnd, ATC_EABS);
    E += (bnd + E + mu_max) * 1.1921e-07f;  // the subtraction of mu: 2 u (|y| + |mu|)
    // the middle tier: 9 u sum |x R| + u (|v| + |mu|), charged 16.8 u bnd + 2 u max |mu|
    const float E2 = __fmaf_rn(1.0e-6f, bnd, __fmaf_rn(1.1921e-07f, mu_max, ATC_EABS));
    float mn = y[0], mx = y[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) {
      mn = fminf(mn, y[i]);
      mx = fmaxf(mx, y[i]);
    }
    s_ex[0][cp][0][m] = mn;
    s_ex[0][cp][1][m] = mx;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + q4), "r"(32 * ATC_PARTS) : "memory");
#pragma unroll
    for (int i = 0; i < ATC_PARTS; ++i) {
      mn = fminf(mn, s_ex[0][i][0][m]);
      mx = fmaxf(mx, s_ex[0][i][1][m]);
    }
    QParams qp;
    const bool q_ok = qparams_certain(mn, mx, E, ro.clip, qp);
    // ---- uncertain scale / zero: the columns that can hold the exact extremes ----
    uint32_t cand = 0u;
    if (valid && !q_ok) {
      const float e2 = 2.0002f * E;
      const float lo_t = __fadd_rn(mn, e2) + fabsf(mn) * P2_M22, hi_t = __fsub_rn(mx, e2) - fabsf(mx) * P2_M22;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (y[i] <= lo_t || y[i] >= hi_t) cand |= 1u << i;
    }
    // the tiers below run only where a row of this lane quarter needs them: the four
    // warps of a quarter hold the same rows, so they agree and meet at the same barriers
    bool q_ok2 = true;
    if (__any_sync(FULLM, valid && !q_ok)) {
      // written for every row: another column part may hold all of a row's candidates
      float m2 = INFINITY, x2 = -INFINITY;
      uint32_t pend = cand;
      while (__any_sync(FULLM, pend != 0u)) {
        float v;
        if (atc_round_f32<F32>(pend, sA, sB, s_mu, 32 * q4, 32 * cp, lane, v) >= 0) {
          m2 = fminf(m2, v);
          x2 = fmaxf(x2, v);
        }
      }
      s_ex[1][cp][0][m] = m2;
      s_ex[1][cp][1][m] = x2;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + q4), "r"(32 * ATC_PARTS) : "memory");
      if (valid && !q_ok) {
        m2 = INFINITY;
        x2 = -INFINITY;
#pragma unroll
        for (int i = 0; i < ATC_PARTS; ++i) {
          m2 = fminf(m2, s_ex[1][i][0][m]);
          x2 = fmaxf(x2, s_ex[1][i][1][m]);
        }
        q_ok2 = qparams_certain(m2, x2, E2, ro.clip, qp);
      }
    }
    if (__any_sync(FULLM, !q_ok2)) {
      DF dmn{INFINITY, 0.f}, dmx{-INFINITY, 0.f};
      uint32_t pend = q_ok2 ? 0u : cand;
      while (__any_sync(FULLM, pend != 0u)) {
        DF v;
        if (atc_round<F32>(pend, sA, sB, s_mu, 32 * q4, 32 * cp, lane, v) >= 0) {
          if (df_less(v, dmn)) dmn = v;
          if (df_less(dmx, v)) dmx = v;
        }
      }
      s_dex[cp][0][m] = make_float2(dmn.hi, dmn.lo);
      s_dex[cp][1][m] = make_float2(dmx.hi, dmx.lo);
      asm volatile("bar.sync %0, %1;" ::"r"(1 + q4), "r"(32 * ATC_PARTS) : "memory");
      if (!q_ok2) {
        DF lo_df{INFINITY, 0.f}, hi_df{-INFINITY, 0.f};
#pragma unroll
        for (int i = 0; i < ATC_PARTS; ++i) {
          const float2 a2 = s_dex[i][0][m], b2 = s_dex[i][1][m];
          if (df_less(DF{a2.x, a2.y}, lo_df)) lo_df = DF{a2.x, a2.y};
          if (df_less(hi_df, DF{b2.x, b2.y})) hi_df = DF{b2.x, b2.y};
        }
        qp = qparams_df(lo_df, hi_df, ro.clip);
      }
    }
    // ---- codes: c = (y - z) / s in paired fp32; |q* - c| <= E / s + 3 u |c| for the
    // exact q* = (x - z) / s, so a code is certain when the clamped c lies further than
    // lim = 0.5 - (E / s + 3.5 u max |c|) from a half-integer ----
    uint32_t packed[2] = {0u, 0u};
    uint32_t unc = 0u;
    if (qp.s > 0.f) {
      const float inv = __frcp_rn(qp.s);
      const float cmax = fmaxf(fabsf(mn - qp.z), fabsf(mx - qp.z)) * inv * 1.0001f;
      const float lim = 0.5f - (E * inv * 1.0001f + cmax * 2.1e-7f);
      const uint64_t pz = f2pk(qp.z, qp.z), pinv = f2pk(inv, inv);
      const uint64_t pmagic = f2pk(12582912.f, 12582912.f);  // 1.5 * 2^23: adding it rounds to an integer
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 cf = f2up(f2mul(f2sub(f2pk(y[2 * i], y[2 * i + 1]), pz), pinv));
        const uint64_t cc = f2pk(fminf(fmaxf(cf.x, 0.f), 3.f), fminf(fmaxf(cf.y, 0.f), 3.f));
        const uint64_t mg = f2add(cc, pmagic);                // the nearest integer in the low mantissa bits
        const float2 f = f2up(f2sub(cc, f2sub(mg, pmagic)));  // c - round(c), exact
        const float2 mgs = f2up(mg);
        packed[i >> 3] |= ((__float_as_uint(mgs.x) & 3u) | ((__float_as_uint(mgs.y) & 3u) << 2)) << (4 * (i & 7));
        if (!(fabsf(f.x) < lim)) unc |= 1u << (2 * i);
        if (!(fabsf(f.y) < lim)) unc |= 1u << (2 * i + 1);
      }
    }
    if (!valid) unc = 0u;
    uint32_t unc3 = 0u;
    while (__any_sync(FULLM, unc != 0u)) {
      float v;
      const int d = atc_round_f32<F32>(unc, sA, sB, s_mu, 32 * q4, 32 * cp, lane, v);
      if (d >= 0) {
        bool c_ok;
        const unsigned c = qcode_certain(v, E2, qp, c_ok);
        if (c_ok) set_code(packed, d, c);
        else unc3 |= 1u << d;
      }
    }
    while (__any_sync(FULLM, unc3 != 0u)) {
      DF v;
      const int d = atc_round<F32>(unc3, sA, sB, s_mu, 32 * q4, 32 * cp, lane, v);
      if (d >= 0) set_code(packed, d, qcode_df(v, qp));
    }
    // ---- write: 8 bytes of codes per thread, the meta by the first part ----
    if (valid) {
      uint8_t* recp = pool + (size_t)s_rec[m] * g.record;
      *reinterpret_cast<uint2*>(recp + ro.codes_off + GROUP_BYTES * s_slot[m] + 8 * cp) =
          make_uint2(packed[0], packed[1]);
      if (cp == 0)
        *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * s_slot[m]) =
            (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
    }
    __syncthreads();  // the unit's items are evaluated and its rows written
    if (u + 1 < u1) prepare(u + 1);
    prefetch(u + 2);  // into this unit's buffer
    issued = early;
  }
  if (!F32) asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy in flight at exit
  if (!alive) {
    // a wait gave up: let the tensor cores finish before tensor memory is freed
    mbar_wait_bounded(&s_bar, phase ^ 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

bool append_dense_tc_supported(int dtype, const void* k, const void* v, const uint8_t* pool) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
                      reinterpret_cast<uintptr_t>(pool);
  return (a & 15u) == 0 && (dtype == KVQ_F32 || dtype == KVQ_BF16);
}

cudaError_t launch_append_dense_tc(const PageGeom& g, int n_seqs, int n_new, int dtype, const int32_t* cu_new,
                                   const int32_t* start_pos, const int32_t* table, const AppendRoles& roles,
                                   int n_roles, uint8_t* pool, unsigned* err, cudaStream_t s) {
  const long long tiles = (n_new + ATC_M - 1) / ATC_M;
  const long long units = (long long)n_roles * g.n_kv_heads * tiles;
  if (units == 0) return cudaSuccess;
  const int grid = (int)std::min<long long>(units, device_sm_count());
  static std::atomic<unsigned long long> attr_bf{0}, attr_f32{0};  // per device
  if (dtype == KVQ_F32) {
    const cudaError_t ea = smem_limit_once(attr_f32, append_dense_tc_kernel<true>, atc_smem_bytes(true));
    if (ea != cudaSuccess) return ea;
    append_dense_tc_kernel<true><<<grid, ATC_THREADS, atc_smem_bytes(true), s>>>(
        g, n_seqs, n_new, cu_new, start_pos, table, roles, n_roles, pool, err);
  } else {
    const cudaError_t ea = smem_limit_once(attr_bf, append_dense_tc_kernel<false>, atc_smem_bytes(false));
    if (ea != cudaSuccess) return ea;
    append_dense_tc_kernel<false><<<grid, ATC_THREADS, atc_smem_bytes(false), s>>>(
        g, n_seqs, n_new, cu_new, start_pos, table, roles, n_roles, pool, err);
  }
  return cudaGetLastError();
}

}  // namespace kvq
