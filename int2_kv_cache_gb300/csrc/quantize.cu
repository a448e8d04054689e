// Write path: key mean, per-head rotation of vectors, and the fused
// rotate -> centre -> clip -> quantize -> pack -> append cache-write kernels.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization": §6 (one cache-write
// launch that rotates keys, subtracts the precomputed mu R, clips, quantizes,
// packs and writes), appendix Eqs. 19-21 (key mean; (k - mu) R = k R - mu R),
// Eq. 27 (values stored rotated), §3.1 Eq. 4 (the quantizer).
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

cudaError_t launch_rotate_heads(int n_rows, int n_heads, int heads_per_rot, const float* x,
                                RotDev rot, float* y, bool transpose, cudaStream_t s) {
  long long warps = (long long)n_rows * n_heads;
  if (warps == 0) return cudaSuccess;
  int blocks = (int)((warps * 32 + 255) / 256);
  rotate_heads_kernel<<<blocks, 256, 0, s>>>(n_rows, n_heads, heads_per_rot, x, rot, y, transpose);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Token -> (sequence, position, physical page, slot) with bounds checks.
// Returns false (and flags) when the token must be skipped.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool locate(int t, int n_seqs, const int32_t* cu_new,
                                       const int32_t* start_pos, const int32_t* table,
                                       const PageGeom& g, unsigned* err, long long* rec_index,
                                       int* slot, int head) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {  // largest b with cu_new[b] <= t
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_new + mid) <= t) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  int base = __ldg(cu_new + b);
  if (t < base || t >= __ldg(cu_new + b + 1)) { flag_error(err, ERR_SEQ_RANGE); return false; }
  long long pos = (long long)__ldg(start_pos + b) + (t - base);
  long long page = pos / g.page_tokens;
  if (pos < 0 || page >= g.max_blocks) { flag_error(err, ERR_POS_RANGE); return false; }
  int blk = __ldg(table + (size_t)b * g.max_blocks + page);
  if (blk < 0 || blk >= g.num_blocks) { flag_error(err, ERR_BLOCK_RANGE); return false; }
  *rec_index = (long long)blk * g.n_kv_heads + head;
  *slot = (int)(pos % g.page_tokens);
  return true;
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

struct AppendRole {
  const void* src;
  RotDev rot;
  const float* mu_rot;
  float clip;
  int codes_off, meta_off;
};
struct AppendRoles {
  AppendRole r[2];
};

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
  if (DENSE) {
    const float4* src = reinterpret_cast<const float4*>(ro.rot.dense + (size_t)h * D * D);
    for (int i = threadIdx.x; i < D * D / 4; i += 256) s_r4[i] = __ldg(src + i);
    __syncthreads();
  }
  for (int t = t0 + warp; t < t1; t += 8) {
    long long rec;
    int slot;
    if (!locate(t, n_seqs, cu_new, start_pos, table, g, err, &rec, &slot, h)) continue;
    const float4 v = load4(ro.src, ((size_t)t * g.n_kv_heads + h) * D + 4 * lane, dtype);
    DF x[4] = {{v.x, 0.f}, {v.y, 0.f}, {v.z, 0.f}, {v.w, 0.f}};
    if (DENSE) dense_rotate_df_smem(x, s_r4, lane);
    else rotate_df_warp(x, ro.rot, h, lane);
    if (ro.mu_rot) {
      const float4 m = __ldg(reinterpret_cast<const float4*>(ro.mu_rot + (size_t)h * D) + lane);
      x[0] = df_add_f(x[0], -m.x); x[1] = df_add_f(x[1], -m.y);
      x[2] = df_add_f(x[2], -m.z); x[3] = df_add_f(x[3], -m.w);
    }
    QParams qp;
    const unsigned byte = quantize_warp_df(x, ro.clip, qp);
    uint8_t* recp = pool + (size_t)rec * g.record;
    recp[ro.codes_off + GROUP_BYTES * slot + lane] = (uint8_t)byte;
    if (lane == 0)
      *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * slot) =
          (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
  }
}

// locate() for one warp: the sequences are searched 32 at a time (one per lane)
// instead of by bisection, so the lookup is a few independent loads deep.
__device__ __forceinline__ bool locate_warp(int t, int n_seqs, const int32_t* cu_new, const int32_t* start_pos,
                                            const int32_t* table, const PageGeom& g, unsigned* err,
                                            long long* rec_index, int* slot, int head, int lane) {
  int b = -1;
  for (int b0 = 0; b0 < n_seqs && b < 0; b0 += 32) {
    const int bb = b0 + lane;
    const bool hit = bb < n_seqs && __ldg(cu_new + bb) <= t && t < __ldg(cu_new + bb + 1);
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) b = b0 + __ffs(m) - 1;
  }
  if (b < 0) {
    if (lane == 0) flag_error(err, ERR_SEQ_RANGE);
    return false;
  }
  const long long pos = (long long)__ldg(start_pos + b) + (t - __ldg(cu_new + b));
  const long long page = pos / g.page_tokens;
  if (pos < 0 || page >= g.max_blocks) {
    if (lane == 0) flag_error(err, ERR_POS_RANGE);
    return false;
  }
  const int blk = __ldg(table + (size_t)b * g.max_blocks + page);
  if (blk < 0 || blk >= g.num_blocks) {
    if (lane == 0) flag_error(err, ERR_BLOCK_RANGE);
    return false;
  }
  *rec_index = (long long)blk * g.n_kv_heads + head;
  *slot = (int)(pos % g.page_tokens);
  return true;
}

// Small appends (a decode step's one token per sequence): one CTA per (token,
// head, role) so the double-float rotations are spread over the whole GPU.
// Warps 0-7 each accumulate the terms of 16 input channels (rows of a dense R_h
// read from global memory, L2-resident, all 16 loads in flight at once) while
// warp 8 finds the token's page slot; the eight double-float partial sums are
// added in a fixed order, and warp 0 centres, quantizes and writes the group.
// grid = (n_new, n_kv_heads, roles), block = 288.
constexpr int APPEND_SMALL_MAX = 128;  // tokens per call below which this path is used

constexpr int APPEND_ROT_WARPS = 8;

__global__ void __launch_bounds__(32 * (APPEND_ROT_WARPS + 1), 2) append_small_dense_kernel(
    PageGeom g, int n_seqs, int dtype, const int32_t* __restrict__ cu_new, const int32_t* __restrict__ start_pos,
    const int32_t* __restrict__ table, AppendRoles roles, uint8_t* __restrict__ pool, unsigned* err) {
  __shared__ float2 part[APPEND_ROT_WARPS][D];  // (hi, lo) of each warp's partial x R
  __shared__ long long s_rec;    // record index, or -1 when the token is skipped
  __shared__ int s_slot;
  const AppendRole ro = blockIdx.z ? roles.r[1] : roles.r[0];
  const int t = blockIdx.x, h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == APPEND_ROT_WARPS) {
    long long rec;
    int slot;
    // flag each bad token once (role 0), skip it in both roles
    const bool ok = locate_warp(t, n_seqs, cu_new, start_pos, table, g, blockIdx.z == 0 ? err : nullptr, &rec, &slot,
                                h, lane);
    if (lane == 0) {
      s_rec = ok ? rec : -1;
      s_slot = slot;
    }
    __syncthreads();
    return;
  }
  const float4 v = load4(ro.src, ((size_t)t * g.n_kv_heads + h) * D + 4 * lane, dtype);
  const float xin[4] = {v.x, v.y, v.z, v.w};
  const float4* R4 = reinterpret_cast<const float4*>(ro.rot.dense + (size_t)h * D * D) + lane;
  float sh[4][4], sl[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i) sh[u][i] = sl[u][i] = 0.f;
  // the warp's 16 rows of R, all loads in flight at once
  {
    float4 rr[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) rr[j] = __ldg(R4 + (size_t)(16 * warp + j) * 32);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int m = 4 * warp + (j >> 2), u = j & 3;          // row 4m + u
      const float xh = __shfl_sync(0xffffffffu, xin[u], m);  // channel 4m + u lives in lane m
      const float r[4] = {rr[j].x, rr[j].y, rr[j].z, rr[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __fmul_rn(xh, r[i]);
        const float pe = __fmaf_rn(xh, r[i], -p);
        const DF q = two_sum(sh[u][i], p);
        sh[u][i] = q.hi;
        sl[u][i] = __fadd_rn(sl[u][i], __fadd_rn(q.lo, pe));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const DF a = df_add(DF{sh[0][i], sl[0][i]}, DF{sh[1][i], sl[1][i]});
    const DF b = df_add(DF{sh[2][i], sl[2][i]}, DF{sh[3][i], sl[3][i]});
    const DF c = df_add(a, b);
    part[warp][4 * lane + i] = make_float2(c.hi, c.lo);
  }
  __syncthreads();
  if (warp != 0) return;
  const long long rec = s_rec;
  const int slot = s_slot;
  if (rec < 0) return;
  DF x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    DF q[APPEND_ROT_WARPS];
#pragma unroll
    for (int w = 0; w < APPEND_ROT_WARPS; ++w) q[w] = DF{part[w][4 * lane + i].x, part[w][4 * lane + i].y};
    x[i] = df_add(df_add(df_add(q[0], q[1]), df_add(q[2], q[3])), df_add(df_add(q[4], q[5]), df_add(q[6], q[7])));
  }
  if (ro.mu_rot) {
    const float4 m = __ldg(reinterpret_cast<const float4*>(ro.mu_rot + (size_t)h * D) + lane);
    x[0] = df_add_f(x[0], -m.x); x[1] = df_add_f(x[1], -m.y);
    x[2] = df_add_f(x[2], -m.z); x[3] = df_add_f(x[3], -m.w);
  }
  QParams qp;
  const unsigned byte = quantize_warp_df(x, ro.clip, qp);
  uint8_t* recp = pool + (size_t)rec * g.record;
  recp[ro.codes_off + GROUP_BYTES * slot + lane] = (uint8_t)byte;
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(recp + ro.meta_off + META_BYTES * slot) =
        (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
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
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(append_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // keys and values may use different rotation kinds: one launch per kind
  const bool kd = rot_k.kind == KVQ_ROT_DENSE, vd = rot_v.kind == KVQ_ROT_DENSE;
  if (n_new <= APPEND_SMALL_MAX && kd && vd) {
    append_small_dense_kernel<<<dim3(n_new, g.n_kv_heads, 2), 32 * (APPEND_ROT_WARPS + 1), 0, s>>>(g, n_seqs, dtype, cu_new, start_pos,
                                                                             table, roles, pool, err);
    return cudaGetLastError();
  }
  if (n_new <= APPEND_SMALL_MAX && (kd || vd)) {
    // dense roles through the small-append kernel, the others through the warp kernel
    for (int role = 0; role < 2; ++role) {
      AppendRoles one;
      one.r[0] = roles.r[role];
      one.r[1] = roles.r[role];
      if (role == 0 ? kd : vd)
        append_small_dense_kernel<<<dim3(n_new, g.n_kv_heads, 1), 32 * (APPEND_ROT_WARPS + 1), 0, s>>>(g, n_seqs, dtype, cu_new, start_pos,
                                                                                 table, one, pool, err);
      else
        append_kernel<false><<<grid, 256, 0, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, one, pool, err);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (kd == vd) {
    const dim3 g2(grid.x, grid.y, 2);
    if (kd) append_kernel<true><<<g2, 256, smem, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, roles, pool, err);
    else append_kernel<false><<<g2, 256, 0, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, roles, pool, err);
    return cudaGetLastError();
  }
  for (int role = 0; role < 2; ++role) {
    AppendRoles one;
    one.r[0] = roles.r[role];
    one.r[1] = roles.r[role];
    if (role == 0 ? kd : vd)
      append_kernel<true><<<grid, 256, smem, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, one, pool, err);
    else
      append_kernel<false><<<grid, 256, 0, s>>>(g, n_seqs, n_new, dtype, cu_new, start_pos, table, one, pool, err);
    const cudaError_t e = cudaGetLastError();
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

}  // namespace kvq
