#include <algorithm>
// Write path: key mean, per-head rotation of vectors, and the fused
// rotate -> centre -> clip -> quantize -> pack -> append cache-write kernels.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization": §6 (one cache-write
// launch that rotates keys, subtracts the precomputed mu R, clips, quantizes,
// packs and writes), appendix Eqs. 19-21 (key mean; (k - mu) R = k R - mu R),
// Eq. 27 (values stored rotated), §3.1 Eq. 4 (the quantizer).
#include <type_traits>

#include "quant_common.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// Eq. 19: mu[h][c] = mean_t k[t][h][c] (fp64 accumulation; one thread per channel).
// ---------------------------------------------------------------------------
__global__ void key_mean_kernel(int n_tok, int n_heads, const void* k, int dtype, float* mu) {
  int h = blockIdx.x;
  int c = threadIdx.x;
  double acc = 0.0;
  for (int t = 0; t < n_tok; ++t) acc += (double)load1(k, ((size_t)t * n_heads + h) * D + c, dtype);
  mu[h * D + c] = (float)(acc / (double)n_tok);
}

cudaError_t launch_key_mean(int n_tok, int n_heads, const void* k, int dtype, float* mu,
                            cudaStream_t s) {
  key_mean_kernel<<<n_heads, D, 0, s>>>(n_tok, n_heads, k, dtype, mu);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// y[r][j] = x[r][j] R_{j/hpr}   (or x R^T when transpose): one warp per vector.
// ---------------------------------------------------------------------------
__global__ void rotate_heads_kernel(int n_rows, int n_heads, int hpr, const float* x, RotDev rot,
                                    float* y, bool transpose) {
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (warp >= n_rows * n_heads) return;
  int j = warp % n_heads;
  float4 v = reinterpret_cast<const float4*>(x + (size_t)warp * D)[lane];
  v = rotate_vec_warp(v, rot, j / hpr, lane, transpose);
  reinterpret_cast<float4*>(y + (size_t)warp * D)[lane] = v;
}

// Dense R, batched: one CTA per (rotation head rh, block of 32 of its n_rows x
// hpr vectors) stages R_rh (or its transpose) in shared memory once; thread t
// forms output channels 4 (t % 32) .. + 3 of vectors t / 32 + 8 i (i < 4).
constexpr int RH_VB = 32;
__global__ void __launch_bounds__(256) rotate_heads_dense_kernel(int n_rows, int n_heads, int hpr, const float* x,
                                                                 const float* __restrict__ dense, float* y,
                                                                 bool transpose) {
  extern __shared__ float rh_smem[];
  float* sR = rh_smem;            // [128][128]: row c = the weights of input channel c
  float* sx = rh_smem + D * D;    // [RH_VB][128]
  const int rh = blockIdx.y, vb0 = blockIdx.x * RH_VB, tid = threadIdx.x;
  const int n_vec = n_rows * hpr;
  const float* R = dense + (size_t)rh * D * D;
  for (int i = tid; i < D * D; i += 256) {
    const int r = i >> 7, c = i & 127;
    sR[i] = transpose ? __ldg(R + (size_t)c * D + r) : __ldg(R + i);
  }
  auto vec_index = [&](int vv) {  // vector vv of this rotation head -> row in x
    const int row = vv / hpr, jj = rh * hpr + vv % hpr;
    return (size_t)row * n_heads + jj;
  };
  for (int i = tid; i < RH_VB * D / 4; i += 256) {
    const int vv = vb0 + i / (D / 4), c4 = i % (D / 4);
    const float4 v = vv < n_vec ? reinterpret_cast<const float4*>(x + vec_index(vv) * D)[c4]
                                : make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(sx + (i / (D / 4)) * D)[c4] = v;
  }
  __syncthreads();
  const int lane = tid & 31, vw = tid >> 5;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int c = 0; c < D; ++c) {
    const float4 r = reinterpret_cast<const float4*>(sR + c * D)[lane];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float xc = sx[(vw + 8 * i) * D + c];
      acc[i].x = fmaf(xc, r.x, acc[i].x); acc[i].y = fmaf(xc, r.y, acc[i].y);
      acc[i].z = fmaf(xc, r.z, acc[i].z); acc[i].w = fmaf(xc, r.w, acc[i].w);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vv = vb0 + vw + 8 * i;
    if (vv < n_vec) reinterpret_cast<float4*>(y + vec_index(vv) * D)[lane] = acc[i];
  }
}

cudaError_t launch_rotate_heads(int n_rows, int n_heads, int heads_per_rot, const float* x,
                                RotDev rot, float* y, bool transpose, cudaStream_t s) {
  long long warps = (long long)n_rows * n_heads;
  if (warps == 0) return cudaSuccess;
  if (rot.kind == KVQ_ROT_DENSE && x != y) {
    constexpr int smem = (D * D + RH_VB * D) * (int)sizeof(float);
    static std::atomic<unsigned long long> attr{0};  // per device
    const cudaError_t ea = smem_limit_once(attr, rotate_heads_dense_kernel, smem);
    if (ea != cudaSuccess) return ea;
    const int n_rot = n_heads / heads_per_rot;
    const int n_vec = n_rows * heads_per_rot;
    rotate_heads_dense_kernel<<<dim3((n_vec + RH_VB - 1) / RH_VB, n_rot), 256, smem, s>>>(
        n_rows, n_heads, heads_per_rot, x, rot.dense, y, transpose);
    return cudaGetLastError();
  }
  int blocks = (int)((warps * 32 + 255) / 256);
  rotate_heads_kernel<<<blocks, 256, 0, s>>>(n_rows, n_heads, heads_per_rot, x, rot, y, transpose);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Cache write: one warp per (token, head) group.  Lane l owns channels 4l..4l+3
// and hence byte l of the packed group.  x = k R - mu R is formed in
// double-float (Eq. 20 with the rotation's rounding errors carried), so the
// quantization decisions are exact.  Keys and values are the two values of
// blockIdx.z; a dense R_h is staged once per CTA in shared memory.
// grid = (ceil(n_new / APPEND_TOK), n_kv_heads, 2), block = 256.
// ---------------------------------------------------------------------------
constexpr int APPEND_TOK = 64;

// x R for a dense R held in shared memory as [128 rows][32 float4], with four
// independent compensated accumulation chains (terms c = 4m + u) per output.
__device__ __forceinline__ void dense_rotate_df_smem(DF x[4], const float4* __restrict__ R4, int lane) {
  float sh[4][4], sl[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i) sh[u][i] = sl[u][i] = 0.f;
#pragma unroll 2
  for (int m = 0; m < 32; ++m) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float xh = __shfl_sync(0xffffffffu, x[u].hi, m);  // channel 4m + u lives in lane m
      const float xl = __shfl_sync(0xffffffffu, x[u].lo, m);
      const float4 r4 = R4[(4 * m + u) * 32 + lane];
      const float r[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __fmul_rn(xh, r[i]);
        float pe = __fmaf_rn(xh, r[i], -p);
        pe = __fmaf_rn(xl, r[i], pe);
        const DF t = two_sum(sh[u][i], p);
        sh[u][i] = t.hi;
        sl[u][i] = __fadd_rn(sl[u][i], __fadd_rn(t.lo, pe));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const DF a = df_add(DF{sh[0][i], sl[0][i]}, DF{sh[1][i], sl[1][i]});
    const DF b = df_add(DF{sh[2][i], sl[2][i]}, DF{sh[3][i], sl[3][i]});
    x[i] = df_add(a, b);
  }
}

template <bool DENSE>
__global__ void __launch_bounds__(256, 1) append_kernel(
    PageGeom g, int n_seqs, int n_new, int dtype, const int32_t* __restrict__ cu_new,
    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ table, AppendRoles roles,
    uint8_t* __restrict__ pool, unsigned* err) {
  extern __shared__ float4 s_r4[];  // dense only: R_h, 128 x 32 float4
  const AppendRole ro = blockIdx.z ? roles.r[1] : roles.r[0];
  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * APPEND_TOK;
  const int t1 = min(n_new, t0 + APPEND_TOK);
  // the tile's tokens are located once, one thread each (record index of head
  // 0 of the token's page, or -1 to skip; slot in the page)
  __shared__ long long s_rec[APPEND_TOK];
  __shared__ int s_slot[APPEND_TOK];
  if (threadIdx.x < APPEND_TOK) {
    const int t = t0 + threadIdx.x;
    long long rec = -1;
    int slot = 0;
    if (t < t1 && !locate(t, n_seqs, cu_new, start_pos, table, g, err, &rec, &slot, 0)) rec = -1;
    s_rec[threadIdx.x] = rec;
    s_slot[threadIdx.x] = slot;
  }
  __shared__ float s_cn[4];  // dense: largest column norm of R_h (from 4 partial maxima)
  if (DENSE) {
    const float4* src = reinterpret_cast<const float4*>(ro.rot.dense + (size_t)h * D * D);
    for (int i = threadIdx.x; i < D * D / 4; i += 256) s_r4[i] = __ldg(src + i);
    __syncthreads();
    // column norms, for the Cauchy-Schwarz bound of the fp32 products below
    if (threadIdx.x < D) {
      const float* sr = reinterpret_cast<const float*>(s_r4);
      float ss = 0.f;
      for (int r = 0; r < D; ++r) ss = fmaf(sr[r * D + threadIdx.x], sr[r * D + threadIdx.x], ss);
      const float cn = warp_max(sqrtf(ss));
      if (lane == 0) s_cn[warp] = cn;
    }
  }
  __syncthreads();
  // largest column norm, with margin for its own rounding
  const float cn_max = DENSE ? fmaxf(fmaxf(s_cn[0], s_cn[1]), fmaxf(s_cn[2], s_cn[3])) * 1.0001f : 0.f;
  for (int t = t0 + warp; t < t1; t += 8) {
    if (s_rec[t - t0] < 0) continue;
    const long long rec = s_rec[t - t0] + h;
    const int slot = s_slot[t - t0];
    const float4 v = load4(ro.src, ((size_t)t * g.n_kv_heads + h) * D + 4 * lane, dtype);
    float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ro.mu_rot) m = __ldg(reinterpret_cast<const float4*>(ro.mu_rot + (size_t)h * D) + lane);
    QParams qp;
    unsigned byte = 0u;
    bool done = false;
    if (!DENSE) {
      // certified fp32 decision (identity and signed Hadamard); a group with an
      // uncertain decision is redone below in double-float
      float y[4] = {v.x, v.y, v.z, v.w};
      float E = rotate_f32_bounded(y, ro.rot, h, lane);
      if (ro.mu_rot) {
        y[0] = __fsub_rn(y[0], m.x); y[1] = __fsub_rn(y[1], m.y);
        y[2] = __fsub_rn(y[2], m.z); y[3] = __fsub_rn(y[3], m.w);
        // the subtraction's rounding: u (|y| + |mu|), y bounded through E's l1 norm or |x|
        E += (warp_max(fmaxf(fmaxf(fabsf(v.x) + fabsf(m.x), fabsf(v.y) + fabsf(m.y)),
                             fmaxf(fabsf(v.z) + fabsf(m.z), fabsf(v.w) + fabsf(m.w)))) +
              E * 524288.f) * P2_M22;
      }
      done = quantize_warp_certain(y, E, ro.clip, qp, byte);
    } else {
      // certified fp32 with a dense R: four FMA chains of 32 terms (channel 4m + u in
      // chain u) and a 2-level sum are off by at most 34.1 u sum_c |x_c R_ci|
      // <= 34.1 u ||x|| ||R_:,i|| (Cauchy-Schwarz): charged 36 u ||x|| max_i ||R_:,i||
      const float xin[4] = {v.x, v.y, v.z, v.w};
      float sh[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) sh[u][i] = 0.f;
#pragma unroll 2
      for (int mm = 0; mm < 32; ++mm) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float xh = __shfl_sync(0xffffffffu, xin[u], mm);  // channel 4mm + u lives in lane mm
          const float4 r4 = s_r4[(4 * mm + u) * 32 + lane];
          sh[u][0] = __fmaf_rn(xh, r4.x, sh[u][0]); sh[u][1] = __fmaf_rn(xh, r4.y, sh[u][1]);
          sh[u][2] = __fmaf_rn(xh, r4.z, sh[u][2]); sh[u][3] = __fmaf_rn(xh, r4.w, sh[u][3]);
        }
      }
      float y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) y[i] = (sh[0][i] + sh[1][i]) + (sh[2][i] + sh[3][i]);
      const float nrm = sqrtf(warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w)) * 1.0001f;
      float E = nrm * cn_max * 2.1458e-06f;  // 36 u
      if (ro.mu_rot) {
        y[0] = __fsub_rn(y[0], m.x); y[1] = __fsub_rn(y[1], m.y);
        y[2] = __fsub_rn(y[2], m.z); y[3] = __fsub_rn(y[3], m.w);
        // the subtraction's rounding: 2 u (|y| + |mu|)
        E += warp_max(fmaxf(fmaxf(fabsf(y[0]) + fabsf(m.x), fabsf(y[1]) + fabsf(m.y)),
                            fmaxf(fabsf(y[2]) + fabsf(m.z), fabsf(y[3]) + fabsf(m.w))) + E) *
             1.1921e-07f;
      }
      done = quantize_warp_certain(y, E, ro.clip, qp, byte);
    }
    if (!done) {
      DF x[4] = {{v.x, 0.f}, {v.y, 0.f}, {v.z, 0.f}, {v.w, 0.f}};
      if (DENSE) dense_rotate_df_smem(x, s_r4, lane);
      else rotate_df_warp(x, ro.rot, h, lane);
      if (ro.mu_rot) {
        x[0] = df_add_f(x[0], -m.x); x[1] = df_add_f(x[1], -m.y);
        x[2] = df_add_f(x[2], -m.z); x[3] = df_add_f(x[3], -m.w);
      }
      byte = quantize_warp_df(x, ro.clip, qp);
    }
    uint8_t* recp = pool + (size_t)rec * g.record;
    recp[ro.codes_off + GROUP_BYTES * slot + lane] = (uint8_t)byte;
    if (lane == 0)
      *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * slot) =
          (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
  }
}

// ---------------------------------------------------------------------------
// Bulk cache write for the identity and signed-Hadamard rotations: certified
// fp32 decisions (quantize_warp_certain's rules) with a double-float redo of
// any group that is not certain.  A warp handles four groups at a time, 8
// lanes x 16 channels each (lane j of a group owns channels 16j..16j+15 and so
// 4 bytes of the packed codes); the Walsh-Hadamard transform runs its four low
// stages in registers and its three high stages across the 8 lanes, and the
// paired fp32 instructions of sm_100 (f32x2) do two channels each.  Groups with
// an uncertain decision are listed in shared memory and redone at the end of
// the CTA, one warp each, in double-float.  Tasks are
// (token, head) in token-major order, so a warp's four groups are consecutive
// input rows.  Per CTA: tpc <= AF_TOK tokens, located once, and per head the sign
// masks and the rotated key mean staged in shared memory.
// grid = (ceil(n_new / tpc), roles), block = AF_THREADS; tpc is chosen so that the CTAs fill
// whole waves of the GPU (four resident CTAs per SM).
// ---------------------------------------------------------------------------
constexpr int AF_TOK = 32;
constexpr int AF_THREADS = 256;
constexpr int AF_MAX_HEADS = 192;  // shared-memory staging: 1,156 bytes per head
constexpr int AF_LPG = 8;          // lanes per group

template <int LPG>  // lanes per group: 8 (16 channels each) or 4 (32)
__global__ void __launch_bounds__(AF_THREADS, 4) append_fast_kernel(
    PageGeom g, int n_seqs, int n_new, int tpc, int dtype, const int32_t* __restrict__ cu_new,
    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ table, AppendRoles roles,
    uint8_t* __restrict__ pool, unsigned* err) {
  constexpr unsigned FULLM = 0xffffffffu;
  constexpr int CPL = D / LPG;   // channels per lane
  constexpr int NP = CPL / 2;    // channel pairs per lane
  constexpr int GPW = 32 / LPG;  // groups (consecutive heads of one token) per warp
  constexpr unsigned GMASK = (1u << LPG) - 1u;
  using Codes = typename std::conditional<LPG == 8, uint32_t, uint64_t>::type;
  constexpr int NQ = CPL / 4;    // 16-byte input words per lane (fp32; bf16 uses the first half)
  constexpr float U1 = 6.5e-8f;  // 1.09 u: one rounding, with margin
  const AppendRole ro = blockIdx.y ? roles.r[1] : roles.r[0];
  const int H = g.n_kv_heads;
  const int t0 = blockIdx.x * tpc;
  const int nt = min(tpc, n_new - t0);
  const bool had = ro.rot.kind == KVQ_ROT_SIGNED_HADAMARD;
  const bool has_mu = ro.mu_rot != nullptr;
  __shared__ long long s_rec[AF_TOK];
  __shared__ int s_slot[AF_TOK];
  __shared__ int s_nredo;
  extern __shared__ uint32_t s_dyn[];
  // per head: sign-bit masks (fp32 input: word c = channel c; bf16: word w = channels 2w, 2w + 1
  // in bits 15 / 31), the rotated key mean (or 0), max |mean|; then the groups to redo
  uint32_t* s_msk = s_dyn;                                  // [H][128]
  float* s_mu = reinterpret_cast<float*>(s_dyn + H * 128);  // [H][128]
  float* s_mumax = s_mu + H * 128;                          // [H]
  int* s_redo = reinterpret_cast<int*>(s_mumax + H);        // [AF_TOK * H]: token << 8 | head
  if (threadIdx.x < nt) {
    const int t = t0 + threadIdx.x;
    long long rec = -1;
    int slot = 0;
    if (t < n_new && !locate(t, n_seqs, cu_new, start_pos, table, g, err, &rec, &slot, 0)) rec = -1;
    s_rec[threadIdx.x] = rec;
    s_slot[threadIdx.x] = slot;
  }
  if (threadIdx.x == 0) s_nredo = 0;
  for (int i = threadIdx.x; i < H * 128; i += AF_THREADS) {
    const int h = i >> 7, c = i & 127;
    const float* sg = ro.rot.signs + (size_t)h * D;
    uint32_t word = 0u;
    if (had) {
      if (dtype == KVQ_F32) word = __ldg(sg + c) < 0.f ? 0x80000000u : 0u;
      else if (c < 64) word = (__ldg(sg + 2 * c) < 0.f ? 0x00008000u : 0u) | (__ldg(sg + 2 * c + 1) < 0.f ? 0x80000000u : 0u);
    }
    s_msk[i] = word;
    s_mu[i] = has_mu ? __ldg(ro.mu_rot + i) : 0.f;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  for (int h = warp; h < H; h += AF_THREADS / 32) {
    const float4 m = *reinterpret_cast<const float4*>(s_mu + h * 128 + 4 * lane);
    const float mx = warp_max(fmaxf(fmaxf(fabsf(m.x), fabsf(m.y)), fmaxf(fabsf(m.z), fabsf(m.w))));
    if (lane == 0) s_mumax[h] = mx;
  }
  __syncthreads();

  const int gq = lane / LPG, j = lane % LPG;
  const uint64_t pinv = f2pk(INV_SQRT_D, INV_SQRT_D);
  const uint64_t pmagic = f2pk(12582912.f, 12582912.f);  // 1.5 * 2^23: adding it rounds to an integer
  const int n_hb = (H + GPW - 1) / GPW;
  // a warp iteration: token tl, heads GPW hb .. GPW hb + GPW - 1
  auto fetch = [&](int tlk, int hbk, uint4 (&raw)[NQ]) {
    const int hk = GPW * hbk + gq;
#pragma unroll
    for (int q = 0; q < NQ; ++q) raw[q] = make_uint4(0u, 0u, 0u, 0u);
    if (tlk < nt && hk < H && s_rec[tlk] >= 0) {
      const size_t rw = ((size_t)(t0 + tlk) * H + hk) * D + CPL * j;
      if (dtype == KVQ_F32) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) raw[q] = __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(ro.src) + rw) + q);
      } else {
#pragma unroll
        for (int q = 0; q < NQ / 2; ++q)
          raw[q] = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ro.src) + rw) + q);
      }
    }
  };
  // warp w takes the (token, head block) pairs w, w + 8, ... (a one-token append still
  // spreads its head blocks over the warps)
  constexpr int NWARP = AF_THREADS / 32;
  const int n_pairs = nt * n_hb;
  const int q8 = NWARP / n_hb, r8 = NWARP - q8 * n_hb;  // the pair step in (token, head block)
  uint4 nxt[NQ];
  int pi = warp;
  int tl = pi / n_hb, hb = pi - tl * n_hb;
  if (pi < n_pairs) fetch(tl, hb, nxt);
  while (pi < n_pairs) {
    uint4 cur[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) cur[q] = nxt[q];
    const int pin = pi + NWARP;
    int tln = tl + q8, hbn = hb + r8;
    if (hbn >= n_hb) {
      hbn -= n_hb;
      ++tln;
    }
    if (pin < n_pairs) fetch(tln, hbn, nxt);
    const int h = GPW * hb + gq;
    const long long rec0 = s_rec[tl];
    const bool live = h < H && rec0 >= 0;
    const int hs = h < H ? h : 0;  // a valid head for the shared-memory tables
    // ---- 16 channels with signs, channel bit 0 butterflies done while unpacking ----
    uint64_t P[NP];
    float l1 = 0.f;
    if (dtype == KVQ_F32) {
      const uint4* mk = reinterpret_cast<const uint4*>(s_msk + hs * 128 + CPL * j);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const uint4 m = mk[q];
        const float ax = __uint_as_float(cur[q].x ^ m.x), ay = __uint_as_float(cur[q].y ^ m.y);
        const float az = __uint_as_float(cur[q].z ^ m.z), aw = __uint_as_float(cur[q].w ^ m.w);
        l1 += (fabsf(ax) + fabsf(ay)) + (fabsf(az) + fabsf(aw));
        if (had) {
          P[2 * q] = f2pk(__fadd_rn(ax, ay), __fsub_rn(ax, ay));
          P[2 * q + 1] = f2pk(__fadd_rn(az, aw), __fsub_rn(az, aw));
        } else {
          P[2 * q] = f2pk(ax, ay);
          P[2 * q + 1] = f2pk(az, aw);
        }
      }
    } else {
      const uint4* mk = reinterpret_cast<const uint4*>(s_msk + hs * 128 + (CPL / 2) * j);
#pragma unroll
      for (int q = 0; q < NQ / 2; ++q) {
        const uint4 m = mk[q];
        const uint32_t ww[4] = {cur[q].x ^ m.x, cur[q].y ^ m.y, cur[q].z ^ m.z, cur[q].w ^ m.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = __uint_as_float(ww[i] << 16), b = __uint_as_float(ww[i] & 0xffff0000u);
          l1 += fabsf(a) + fabsf(b);
          P[4 * q + i] = had ? f2pk(__fadd_rn(a, b), __fsub_rn(a, b)) : f2pk(a, b);
        }
      }
    }
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) l1 += __shfl_xor_sync(FULLM, l1, m);
    // ---- rotation, with a bound E on |y - (x R)| for every channel of the group ----
    float E = 0.f, ymax = l1;  // identity: exact, |y| <= l1
    if (had) {
#pragma unroll
      for (int b = 1; b < NP; b <<= 1)  // channel bits 1-3 (between pairs)
#pragma unroll
        for (int i = 0; i < NP; ++i)
          if (!(i & b)) {
            const uint64_t a = P[i], c = P[i | b];
            P[i] = f2add(a, c);
            P[i | b] = f2sub(a, c);
          }
      // channel bits 4-6 (lanes j ^ 1, 2, 4): lower half y + p, upper half p - y
#pragma unroll
      for (int m = 1; m < LPG; m <<= 1) {
        const float sgn = (j & m) ? -1.f : 1.f;
        const uint64_t sp = f2pk(sgn, sgn);
#pragma unroll
        for (int i = 0; i < NP; ++i) P[i] = f2fma(sp, P[i], __shfl_xor_sync(FULLM, P[i], m));
      }
#pragma unroll
      for (int i = 0; i < NP; ++i) P[i] = f2mul(P[i], pinv);
      // each stage adds at most u * l1 to an output (the nodes an output depends on
      // at one stage partition the inputs): 7 u l1; the scaling by fp32(1/sqrt(128))
      // (relative error < 0.2 u) and its rounding (u |y|, |y| <= l1 / sqrt(128)): 8.2 u
      ymax = l1 * INV_SQRT_D;
      E = ymax * 5.1e-7f;  // 8.56 u
    }
    if (has_mu) {
      const uint64_t* mp = reinterpret_cast<const uint64_t*>(s_mu + hs * 128 + CPL * j);
#pragma unroll
      for (int i = 0; i < NP; ++i) P[i] = f2sub(P[i], mp[i]);
      E = __fmaf_rn(ymax + s_mumax[hs], U1, E);  // rounding of y - mu
    }
    // ---- group decision (certified) ----
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const float2 v = f2up(P[i]);
      mn = fminf(mn, fminf(v.x, v.y));
      mx = fmaxf(mx, fmaxf(v.x, v.y));
    }
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULLM, mn, m));
      mx = fmaxf(mx, __shfl_xor_sync(FULLM, mx, m));
    }
    const float clip = ro.clip;
    const float lo = __fmul_rn(clip, mn), hi = __fmul_rn(clip, mx);
    const float elo = __fmaf_rn(clip, E, fabsf(lo) * U1);
    const float ehi = __fmaf_rn(clip, E, fabsf(hi) * U1);
    const float range = __fsub_rn(hi, lo);
    const float third = __fdiv_rn(range, 3.0f);
    const float eth = (elo + ehi + fabsf(range) * U1) * 0.33334f + fabsf(third) * U1;
    __half s16, z16;
    bool ok = half_rn_certain(third, eth, s16);
    ok = half_rn_certain(lo, elo, z16) && ok;
    const float sc = __half2float(s16), zf = __half2float(z16);
    Codes codes = 0u;
    if (sc > 0.f) {
      const float inv = __frcp_rn(sc);
      // |q* - c| <= E / s + 3 u |c| for c = fl(fl(d - z) / s) and q* = (x - z) / s;
      // a code is certain when the clamped c is further than that from a half-integer
      const float cmax = fmaxf(fabsf(mn - zf), fabsf(mx - zf)) * inv * 1.0001f;
      const float lim = 0.5f - (E * inv * 1.0001f + cmax * 2.1e-7f);  // 3.5 u
      const uint64_t pz = f2pk(zf, zf), pinv2 = f2pk(inv, inv);
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const float2 cf = f2up(f2mul(f2sub(P[i], pz), pinv2));
        const uint64_t cc = f2pk(fminf(fmaxf(cf.x, 0.f), 3.f), fminf(fmaxf(cf.y, 0.f), 3.f));
        const uint64_t mg = f2add(cc, pmagic);                   // integer r in the low mantissa bits
        const float2 f = f2up(f2sub(cc, f2sub(mg, pmagic)));     // c - r, exact
        ok = ok && fabsf(f.x) < lim && fabsf(f.y) < lim;
        const float2 mgs = f2up(mg);
        codes |= (Codes)((__float_as_uint(mgs.x) & 3u) | ((__float_as_uint(mgs.y) & 3u) << 2)) << (4 * i);
      }
    }
    const unsigned bad = __ballot_sync(FULLM, live && !ok);
    const int slot = s_slot[tl];
    if (live && ((bad >> (LPG * gq)) & GMASK) == 0u) {
      uint8_t* recp = pool + (size_t)(rec0 + h) * g.record;
      *reinterpret_cast<Codes*>(recp + ro.codes_off + GROUP_BYTES * slot + (CPL / 4) * j) = codes;
      if (j == 0)
        *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * slot) =
            (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
    }
    // groups with an uncertain decision are listed and redone after the loop
    if (live && j == 0 && ((bad >> (LPG * gq)) & GMASK) != 0u) s_redo[atomicAdd(&s_nredo, 1)] = (tl << 8) | h;
    pi = pin;
    tl = tln;
    hb = hbn;
  }
  // ---- the listed groups: one warp each, in double-float ----
  __syncthreads();
  for (int i = warp; i < s_nredo; i += AF_THREADS / 32) {
    const int tlq = s_redo[i] >> 8, hq = s_redo[i] & 0xff;
    const float4 v = load4(ro.src, ((size_t)(t0 + tlq) * H + hq) * D + 4 * lane, dtype);
    DF x[4] = {{v.x, 0.f}, {v.y, 0.f}, {v.z, 0.f}, {v.w, 0.f}};
    rotate_df_warp(x, ro.rot, hq, lane);
    if (has_mu) {
      const float4 m = *reinterpret_cast<const float4*>(s_mu + hq * 128 + 4 * lane);
      x[0] = df_add_f(x[0], -m.x); x[1] = df_add_f(x[1], -m.y);
      x[2] = df_add_f(x[2], -m.z); x[3] = df_add_f(x[3], -m.w);
    }
    QParams qp;
    const unsigned byte = quantize_warp_df(x, ro.clip, qp);
    uint8_t* recp = pool + (size_t)(s_rec[tlq] + hq) * g.record;
    recp[ro.codes_off + GROUP_BYTES * s_slot[tlq] + lane] = (uint8_t)byte;
    if (lane == 0)
      *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * s_slot[tlq]) =
          (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
  }
}

constexpr int APPEND_SMALL_MAX = 128;  // tokens per call below which the step kernel is used

// ---------------------------------------------------------------------------
// Cache write with a dense R for a few tokens (a decode step): one CTA per
// (tb <= ADS_TB tokens, head, role), 8 warps.  Warp w keeps rows 16w..16w+15 of R_h in
// registers and forms, for every token of the CTA, its partial x R and the
// partial sum of |x_c| |R_ci| (the error bound's scale).  Warp t then adds the
// 8 partials of token t in a fixed tree and decides the group with certified
// fp32 (quantize_warp_certain): a 16-term FMA chain and a 3-level sum are off
// by at most 19.1 u sum_c |x_c R_ci|.  Uncertain groups are redone by all 8
// warps in double-float from the same register-held rows.
// grid = (ceil(n_new / tb), n_kv_heads, roles), block = 256, tb chosen for ~2 CTAs per SM.
// ---------------------------------------------------------------------------
constexpr int ADS_TB = 8;

__global__ void __launch_bounds__(256) append_dense_step_kernel(
    PageGeom g, int n_seqs, int n_new, int tb, int dtype, const int32_t* __restrict__ cu_new,
    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ table, AppendRoles roles,
    uint8_t* __restrict__ pool, unsigned* err) {
  __shared__ __align__(16) float s_x[ADS_TB][D];          // the tokens' input rows
  __shared__ __align__(16) float4 s_val[ADS_TB][8][32];   // partial x R (lane l: outputs 4l..4l+3)
  __shared__ float s_abs[ADS_TB][8];                      // max over the warp's outputs of its partial sum |x| |R|
  __shared__ long long s_rec[ADS_TB];
  __shared__ int s_slot[ADS_TB], s_redo[ADS_TB];
  const AppendRole ro = blockIdx.z ? roles.r[1] : roles.r[0];
  const int h = blockIdx.y, t0 = blockIdx.x * tb;
  const int nt = min(tb, n_new - t0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // rows 16 warp .. 16 warp + 15 of R_h, lane l: columns 4l .. 4l + 3 (issued first: the
  // token lookups and input loads below overlap them)
  const float4* R4 = reinterpret_cast<const float4*>(ro.rot.dense + (size_t)h * D * D) + lane;
  float4 rr[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) rr[r] = __ldg(R4 + (size_t)(16 * warp + r) * 32);
  for (int i = warp; i < ADS_TB; i += 8) {
    const float4 v = i < nt ? load4(ro.src, ((size_t)(t0 + i) * g.n_kv_heads + h) * D + 4 * lane, dtype)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(s_x[i])[lane] = v;
  }
  if (warp == 7 && lane < ADS_TB) {
    const int t = t0 + lane;
    long long rec = -1;
    int slot = 0;
    // each bad token is flagged once (role 0) and skipped in both roles
    if (lane < nt && !locate(t, n_seqs, cu_new, start_pos, table, g, blockIdx.z == 0 ? err : nullptr, &rec, &slot, h))
      rec = -1;
    s_rec[lane] = rec;
    s_slot[lane] = slot;
    s_redo[lane] = 0;
  }
  __syncthreads();
  for (int tk = 0; tk < nt; ++tk) {
    float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float xc = s_x[tk][16 * warp + r], ax = fabsf(xc);
      a[0] = __fmaf_rn(xc, rr[r].x, a[0]); a[1] = __fmaf_rn(xc, rr[r].y, a[1]);
      a[2] = __fmaf_rn(xc, rr[r].z, a[2]); a[3] = __fmaf_rn(xc, rr[r].w, a[3]);
      b[0] = __fmaf_rn(ax, fabsf(rr[r].x), b[0]); b[1] = __fmaf_rn(ax, fabsf(rr[r].y), b[1]);
      b[2] = __fmaf_rn(ax, fabsf(rr[r].z), b[2]); b[3] = __fmaf_rn(ax, fabsf(rr[r].w), b[3]);
    }
    s_val[tk][warp][lane] = make_float4(a[0], a[1], a[2], a[3]);
    const float bm = warp_max(fmaxf(fmaxf(b[0], b[1]), fmaxf(b[2], b[3])));
    if (lane == 0) s_abs[tk][warp] = bm;
  }
  __syncthreads();
  float4 mu = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ro.mu_rot) mu = __ldg(reinterpret_cast<const float4*>(ro.mu_rot + (size_t)h * D) + lane);
  if (warp < nt && s_rec[warp] >= 0) {
    const int tk = warp;
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 p = s_val[tk][w][lane];
        v[w] = i == 0 ? p.x : i == 1 ? p.y : i == 2 ? p.z : p.w;
      }
      y[i] = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    }
    // sum over warps of each warp's largest partial sum |x R| bounds every output's
    // sum_c |x_c R_ci|; 16-term chains and a 3-level sum are off by at most 19.1 u of
    // it, and the computed bound is itself low by at most 20 u: 20 u * 1.0001 covers both
    const float bound = ((s_abs[tk][0] + s_abs[tk][1]) + (s_abs[tk][2] + s_abs[tk][3])) +
                        ((s_abs[tk][4] + s_abs[tk][5]) + (s_abs[tk][6] + s_abs[tk][7]));
    float E = bound * 1.1921e-06f;  // 20 u
    if (ro.mu_rot) {
      y[0] = __fsub_rn(y[0], mu.x); y[1] = __fsub_rn(y[1], mu.y);
      y[2] = __fsub_rn(y[2], mu.z); y[3] = __fsub_rn(y[3], mu.w);
      E += warp_max(fmaxf(fmaxf(fabsf(y[0]) + fabsf(mu.x), fabsf(y[1]) + fabsf(mu.y)),
                          fmaxf(fabsf(y[2]) + fabsf(mu.z), fabsf(y[3]) + fabsf(mu.w))) + E) *
           1.1921e-07f;  // rounding of y - mu (2 u)
    }
    QParams qp;
    unsigned byte = 0u;
    if (quantize_warp_certain(y, E, ro.clip, qp, byte)) {
      uint8_t* recp = pool + (size_t)s_rec[tk] * g.record;
      recp[ro.codes_off + GROUP_BYTES * s_slot[tk] + lane] = (uint8_t)byte;
      if (lane == 0)
        *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * s_slot[tk]) =
            (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
    } else if (lane == 0) {
      s_redo[tk] = 1;
    }
  }
  __syncthreads();
  // ---- double-float redo of the uncertain groups, all warps ----
  float2* part = reinterpret_cast<float2*>(&s_val[0][0][0]);  // [8 warps][128] (hi, lo)
  for (int tk = 0; tk < nt; ++tk) {
    if (!s_redo[tk]) continue;  // uniform: shared flag after a barrier
    float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float xc = s_x[tk][16 * warp + r];
      const float rv[4] = {rr[r].x, rr[r].y, rr[r].z, rr[r].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __fmul_rn(xc, rv[i]);
        const float pe = __fmaf_rn(xc, rv[i], -p);
        const DF q = two_sum(sh[i], p);
        sh[i] = q.hi;
        sl[i] = __fadd_rn(sl[i], __fadd_rn(q.lo, pe));
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const DF c = df_norm(sh[i], sl[i]);
      part[warp * D + 4 * lane + i] = make_float2(c.hi, c.lo);
    }
    __syncthreads();
    if (warp == 0) {
      DF x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        DF q[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) q[w] = DF{part[w * D + 4 * lane + i].x, part[w * D + 4 * lane + i].y};
        x[i] = df_add(df_add(df_add(q[0], q[1]), df_add(q[2], q[3])), df_add(df_add(q[4], q[5]), df_add(q[6], q[7])));
      }
      if (ro.mu_rot) {
        x[0] = df_add_f(x[0], -mu.x); x[1] = df_add_f(x[1], -mu.y);
        x[2] = df_add_f(x[2], -mu.z); x[3] = df_add_f(x[3], -mu.w);
      }
      QParams qp;
      const unsigned byte = quantize_warp_df(x, ro.clip, qp);
      uint8_t* recp = pool + (size_t)s_rec[tk] * g.record;
      recp[ro.codes_off + GROUP_BYTES * s_slot[tk] + lane] = (uint8_t)byte;
      if (lane == 0)
        *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * s_slot[tk]) =
            (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
    }
    __syncthreads();
  }
}

// Tokens per CTA of append_dense_step_kernel: about 300 CTAs (two per SM), at most ADS_TB.
static int dense_step_tokens(int n_new, int n_heads, int n_roles) {
  const long long groups = (long long)n_new * n_heads * n_roles;
  long long tb = (groups + 299) / 300;
  if (tb < 1) tb = 1;
  if (tb > ADS_TB) tb = ADS_TB;
  return (int)tb;
}

// Non-dense roles: the certified kernel (the warp-per-group kernel beyond AF_MAX_HEADS heads).
static cudaError_t launch_append_nondense(const PageGeom& g, int n_seqs, int n_new, int dtype, const int32_t* cu_new,
                                          const int32_t* start_pos, const int32_t* table, const AppendRoles& roles,
                                          int n_roles, uint8_t* pool, unsigned* err, cudaStream_t s) {
  if (g.n_kv_heads > AF_MAX_HEADS) {
    const dim3 grid((n_new + APPEND_TOK - 1) / APPEND_TOK, g.n_kv_heads, n_roles);
    append_kernel<false><<<grid, 256, 0, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, roles, pool, err);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)g.n_kv_heads * (1028 + 4 * AF_TOK);
  static std::atomic<unsigned long long> attr_set{0};  // per device
  const cudaError_t ea = smem_limit_once(attr_set, append_fast_kernel<AF_LPG>, AF_MAX_HEADS * (1028 + 4 * AF_TOK));
  if (ea != cudaSuccess) return ea;
  // tokens per CTA: fill whole waves (four resident CTAs per SM) instead of leaving a partial one
  const long long slots = 4LL * device_sm_count();
  const long long waves = ((long long)(n_new + AF_TOK - 1) / AF_TOK * n_roles + slots - 1) / slots;
  const int tpc = (int)std::min<long long>(AF_TOK, std::max<long long>(1, ((long long)n_new * n_roles + waves * slots - 1) / (waves * slots)));
  append_fast_kernel<AF_LPG><<<dim3((n_new + tpc - 1) / tpc, n_roles), AF_THREADS, smem, s>>>(
      g, n_seqs, n_new, tpc, dtype, cu_new, start_pos, table, roles, pool, err);
  return cudaGetLastError();
}

cudaError_t launch_quantize_append(const PageGeom& g, int n_seqs, int n_new, const void* k,
                                   const void* v, int dtype, const int32_t* cu_new,
                                   const int32_t* start_pos, const int32_t* table, RotDev rot_k,
                                   RotDev rot_v, const float* mu_rot_k, float clip_k, float clip_v,
                                   uint8_t* pool, unsigned* err, cudaStream_t s) {
  if (n_new == 0) return cudaSuccess;
  const int P = g.page_tokens;
  AppendRoles roles;
  roles.r[0] = AppendRole{k, rot_k, mu_rot_k, clip_k, 0, 64 * P};
  roles.r[1] = AppendRole{v, rot_v, nullptr, clip_v, 32 * P, 68 * P};
  const dim3 grid((n_new + APPEND_TOK - 1) / APPEND_TOK, g.n_kv_heads, 1);
  const size_t smem = (size_t)D * D * sizeof(float);
  static std::atomic<unsigned long long> attr_set{0};  // per device
  const cudaError_t ea = smem_limit_once(attr_set, append_kernel<true>, (int)smem);
  if (ea != cudaSuccess) return ea;
  // keys and values may use different rotation kinds: one launch per kind
  const bool kd = rot_k.kind == KVQ_ROT_DENSE, vd = rot_v.kind == KVQ_ROT_DENSE;
  if (!kd && !vd) return launch_append_nondense(g, n_seqs, n_new, dtype, cu_new, start_pos, table, roles, 2, pool, err, s);
  if (n_new <= APPEND_SMALL_MAX && kd && vd) {
    const int tb = dense_step_tokens(n_new, g.n_kv_heads, 2);
    append_dense_step_kernel<<<dim3((n_new + tb - 1) / tb, g.n_kv_heads, 2), 256, 0, s>>>(
        g, n_seqs, n_new, tb, dtype, cu_new, start_pos, table, roles, pool, err);
    return cudaGetLastError();
  }
  // chunks beyond a decode step: the tensor-core kernel (the fp32 FMA kernel for unaligned inputs)
  const bool tc = append_dense_tc_supported(dtype, k, v, pool);
  if (kd && vd) {
    if (tc) return launch_append_dense_tc(g, n_seqs, n_new, dtype, cu_new, start_pos, table, roles, 2, pool, err, s);
    append_kernel<true><<<dim3(grid.x, grid.y, 2), 256, smem, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table,
                                                                     roles, pool, err);
    return cudaGetLastError();
  }
  // one dense role and one other
  for (int role = 0; role < 2; ++role) {
    AppendRoles one;
    one.r[0] = roles.r[role];
    one.r[1] = roles.r[role];
    cudaError_t e;
    if (role == 0 ? kd : vd) {
      if (n_new <= APPEND_SMALL_MAX)
        append_dense_step_kernel<<<dim3((n_new + dense_step_tokens(n_new, g.n_kv_heads, 1) - 1) /
                                            dense_step_tokens(n_new, g.n_kv_heads, 1),
                                        g.n_kv_heads, 1),
                                   256, 0, s>>>(g, n_seqs, n_new, dense_step_tokens(n_new, g.n_kv_heads, 1), dtype,
                                                cu_new, start_pos, table, one, pool, err);
      else if (tc) {
        e = launch_append_dense_tc(g, n_seqs, n_new, dtype, cu_new, start_pos, table, one, 1, pool, err, s);
        if (e != cudaSuccess) return e;
      } else
        append_kernel<true><<<grid, 256, smem, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, one, pool, err);
      e = cudaGetLastError();
    } else {
      e = launch_append_nondense(g, n_seqs, n_new, dtype, cu_new, start_pos, table, one, 1, pool, err, s);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Calibration helpers.
// rotate_df: x = (src - mu) R per (row, head), kept as double-float (hi, lo planes).
// quant_dequant_df: out = zero + scale * code of each group of x.
// One warp per group.
// ---------------------------------------------------------------------------
__global__ void rotate_df_kernel(int n_rows, int n_heads, const void* __restrict__ src, int dtype,
                                 const float* __restrict__ mu, RotDev rot, float* __restrict__ x_hi,
                                 float* __restrict__ x_lo) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_rows * n_heads) return;
  const int h = w % n_heads;
  const float4 v = load4(src, (size_t)w * D + 4 * lane, dtype);
  DF x[4] = {{v.x, 0.f}, {v.y, 0.f}, {v.z, 0.f}, {v.w, 0.f}};
  if (mu) {
    const float4 m = __ldg(reinterpret_cast<const float4*>(mu + (size_t)h * D) + lane);
    x[0] = two_sum(v.x, -m.x); x[1] = two_sum(v.y, -m.y);
    x[2] = two_sum(v.z, -m.z); x[3] = two_sum(v.w, -m.w);
  }
  rotate_df_warp(x, rot, h, lane);
  reinterpret_cast<float4*>(x_hi + (size_t)w * D)[lane] = make_float4(x[0].hi, x[1].hi, x[2].hi, x[3].hi);
  reinterpret_cast<float4*>(x_lo + (size_t)w * D)[lane] = make_float4(x[0].lo, x[1].lo, x[2].lo, x[3].lo);
}

cudaError_t launch_rotate_df(int n_rows, int n_heads, const void* src, int dtype, const float* mu,
                             RotDev rot, float* x_hi, float* x_lo, cudaStream_t s) {
  const long long warps = (long long)n_rows * n_heads;
  if (warps == 0) return cudaSuccess;
  rotate_df_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, s>>>(n_rows, n_heads, src, dtype, mu, rot,
                                                                      x_hi, x_lo);
  return cudaGetLastError();
}

__global__ void quant_dequant_df_kernel(int n_groups, const float* __restrict__ x_hi,
                                        const float* __restrict__ x_lo, float clip,
                                        float* __restrict__ out) {
  const int gi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gi >= n_groups) return;
  const float4 a = reinterpret_cast<const float4*>(x_hi + (size_t)gi * D)[lane];
  const float4 b = reinterpret_cast<const float4*>(x_lo + (size_t)gi * D)[lane];
  const DF x[4] = {{a.x, b.x}, {a.y, b.y}, {a.z, b.z}, {a.w, b.w}};
  QParams qp;
  const unsigned byte = quantize_warp_df(x, clip, qp);
  float4 o;
  o.x = fmaf(qp.s, (float)(byte & 3u), qp.z);
  o.y = fmaf(qp.s, (float)((byte >> 2) & 3u), qp.z);
  o.z = fmaf(qp.s, (float)((byte >> 4) & 3u), qp.z);
  o.w = fmaf(qp.s, (float)((byte >> 6) & 3u), qp.z);
  reinterpret_cast<float4*>(out + (size_t)gi * D)[lane] = o;
}

cudaError_t launch_quant_dequant(int n_groups, const float* x_hi, const float* x_lo, float clip,
                                 float* out, cudaStream_t s) {
  if (n_groups == 0) return cudaSuccess;
  const int blocks = (int)(((long long)n_groups * 32 + 255) / 256);
  quant_dequant_df_kernel<<<blocks, 256, 0, s>>>(n_groups, x_hi, x_lo, clip, out);
  return cudaGetLastError();
}

// quant_to_pool: the same exact group decisions as quant_dequant, packed into the
// records of a private page pool (16-token pages, page t / 16 of the head's record
// row, slot t % 16; role 0 keys, 1 values) instead of dequantized.  One warp per group.
__global__ void quant_pool_df_kernel(int n_groups, int n_kv_heads, const float* __restrict__ x_hi,
                                     const float* __restrict__ x_lo, float clip, int role, uint8_t* __restrict__ pool) {
  constexpr int P = CALIB_PAGE;
  const int gi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gi >= n_groups) return;
  const float4 a = reinterpret_cast<const float4*>(x_hi + (size_t)gi * D)[lane];
  const float4 b = reinterpret_cast<const float4*>(x_lo + (size_t)gi * D)[lane];
  const DF x[4] = {{a.x, b.x}, {a.y, b.y}, {a.z, b.z}, {a.w, b.w}};
  QParams qp;
  const unsigned byte = quantize_warp_df(x, clip, qp);
  const int t = gi / n_kv_heads, h = gi % n_kv_heads;
  uint8_t* rec = pool + ((size_t)(t / P) * n_kv_heads + h) * (72 * P);
  rec[(role ? 32 * P : 0) + GROUP_BYTES * (t % P) + lane] = (uint8_t)byte;
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(rec + (role ? 68 * P : 64 * P) + META_BYTES * (t % P)) =
        (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
}

cudaError_t launch_quant_to_pool(int n_tok, int n_kv_heads, const float* x_hi, const float* x_lo, float clip,
                                 int role, uint8_t* pool, cudaStream_t s) {
  const long long n_groups = (long long)n_tok * n_kv_heads;
  if (n_groups == 0) return cudaSuccess;
  quant_pool_df_kernel<<<(unsigned)((n_groups * 32 + 255) / 256), 256, 0, s>>>((int)n_groups, n_kv_heads, x_hi, x_lo,
                                                                                 clip, role, pool);
  return cudaGetLastError();
}

}  // namespace kvq
