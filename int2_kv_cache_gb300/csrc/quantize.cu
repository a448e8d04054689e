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
// Identity / signed-Hadamard cache write: one thread per (token, head) group,
// the 128 values and the Walsh-Hadamard transform held in registers.
// grid = (ceil(n_new / 128), n_kv_heads), block = 128.
// ---------------------------------------------------------------------------
template <int DTYPE, bool HADAMARD>
__global__ void __launch_bounds__(128) append_fwht_kernel(
    PageGeom g, int n_seqs, int n_new, const void* __restrict__ src,
    const int32_t* __restrict__ cu_new, const int32_t* __restrict__ start_pos,
    const int32_t* __restrict__ table, const float* __restrict__ signs,
    const float* __restrict__ mu_rot, float clip, int codes_off, int meta_off,
    uint8_t* __restrict__ pool, unsigned* err) {
  const int h = blockIdx.y;
  __shared__ float s_sign[D];
  __shared__ float s_mu[D];
  s_sign[threadIdx.x] = HADAMARD ? signs[(size_t)h * D + threadIdx.x] : 1.f;
  s_mu[threadIdx.x] = mu_rot ? mu_rot[(size_t)h * D + threadIdx.x] : 0.f;
  __syncthreads();
  const int t = blockIdx.x * 128 + threadIdx.x;
  if (t >= n_new) return;
  long long rec;
  int slot;
  if (!locate(t, n_seqs, cu_new, start_pos, table, g, err, &rec, &slot, h)) return;

  float x[D];
  const size_t row = ((size_t)t * g.n_kv_heads + h) * D;
  if (DTYPE == KVQ_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + row);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float4 f = __ldg(p + i);
      x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + row);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint4 w = __ldg(p + i);
      x[8 * i + 0] = __uint_as_float(w.x << 16); x[8 * i + 1] = __uint_as_float(w.x & 0xFFFF0000u);
      x[8 * i + 2] = __uint_as_float(w.y << 16); x[8 * i + 3] = __uint_as_float(w.y & 0xFFFF0000u);
      x[8 * i + 4] = __uint_as_float(w.z << 16); x[8 * i + 5] = __uint_as_float(w.z & 0xFFFF0000u);
      x[8 * i + 6] = __uint_as_float(w.w << 16); x[8 * i + 7] = __uint_as_float(w.w & 0xFFFF0000u);
    }
  }
  float scale = 1.f;
  if (HADAMARD) {
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] *= s_sign[i];
#pragma unroll
    for (int hs = 1; hs < D; hs <<= 1) {
#pragma unroll
      for (int i = 0; i < D; ++i) {
        if ((i & hs) == 0) {
          float a = x[i], b = x[i + hs];
          x[i] = a + b;
          x[i + hs] = a - b;
        }
      }
    }
    scale = INV_SQRT_D;
  }
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < D; ++i) {
    x[i] = fmaf(x[i], scale, -s_mu[i]);
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
  const QParams qp = qparams(mn, mx, clip);
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t acc = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc |= qcode(x[16 * k + j], qp) << (2 * j);
    w[k] = acc;
  }
  uint8_t* recp = pool + (size_t)rec * g.record;
  uint4* dst = reinterpret_cast<uint4*>(recp + codes_off + GROUP_BYTES * slot);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  *reinterpret_cast<uint32_t*>(recp + meta_off + META_BYTES * slot) =
      (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
}

// ---------------------------------------------------------------------------
// Dense-R cache write: one warp per (token, head) group; lane l owns channels
// 4l..4l+3 and hence byte l of the packed group.
// grid = (ceil(n_new / 8), n_kv_heads), block = 256.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) append_dense_kernel(
    PageGeom g, int n_seqs, int n_new, const void* __restrict__ src, int dtype,
    const int32_t* __restrict__ cu_new, const int32_t* __restrict__ start_pos,
    const int32_t* __restrict__ table, RotDev rot, const float* __restrict__ mu_rot, float clip,
    int codes_off, int meta_off, uint8_t* __restrict__ pool, unsigned* err) {
  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= n_new) return;
  long long rec;
  int slot;
  if (!locate(t, n_seqs, cu_new, start_pos, table, g, err, &rec, &slot, h)) return;
  float4 v = load4(src, ((size_t)t * g.n_kv_heads + h) * D + 4 * lane, dtype);
  v = rotate_vec_warp(v, rot, h, lane, false);
  if (mu_rot) {
    float4 m = __ldg(reinterpret_cast<const float4*>(mu_rot + (size_t)h * D) + lane);
    v.x -= m.x; v.y -= m.y; v.z -= m.z; v.w -= m.w;
  }
  float mn = warp_min(fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
  float mx = warp_max(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
  const QParams qp = qparams(mn, mx, clip);
  unsigned byte = qcode(v.x, qp) | (qcode(v.y, qp) << 2) | (qcode(v.z, qp) << 4) | (qcode(v.w, qp) << 6);
  uint8_t* recp = pool + (size_t)rec * g.record;
  recp[codes_off + GROUP_BYTES * slot + lane] = (uint8_t)byte;
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(recp + meta_off + META_BYTES * slot) =
        (uint32_t)qp.s_bits | ((uint32_t)qp.z_bits << 16);
}

cudaError_t launch_quantize_append(const PageGeom& g, int n_seqs, int n_new, const void* src,
                                   int dtype, const int32_t* cu_new, const int32_t* start_pos,
                                   const int32_t* table, RotDev rot, const float* mu_rot,
                                   float clip, int codes_off, int meta_off, uint8_t* pool,
                                   unsigned* err, cudaStream_t s) {
  if (n_new == 0) return cudaSuccess;
  if (rot.kind == KVQ_ROT_DENSE) {
    dim3 grid((n_new + 7) / 8, g.n_kv_heads);
    append_dense_kernel<<<grid, 256, 0, s>>>(g, n_seqs, n_new, src, dtype, cu_new, start_pos,
                                             table, rot, mu_rot, clip, codes_off, meta_off, pool,
                                             err);
    return cudaGetLastError();
  }
  dim3 grid((n_new + 127) / 128, g.n_kv_heads);
  const bool had = rot.kind == KVQ_ROT_SIGNED_HADAMARD;
#define KVQ_LAUNCH(DT, HAD)                                                                   \
  append_fwht_kernel<DT, HAD><<<grid, 128, 0, s>>>(g, n_seqs, n_new, src, cu_new, start_pos, \
                                                   table, rot.signs, mu_rot, clip, codes_off, \
                                                   meta_off, pool, err)
  if (dtype == KVQ_F32) {
    if (had) KVQ_LAUNCH(KVQ_F32, true); else KVQ_LAUNCH(KVQ_F32, false);
  } else {
    if (had) KVQ_LAUNCH(KVQ_BF16, true); else KVQ_LAUNCH(KVQ_BF16, false);
  }
#undef KVQ_LAUNCH
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Quantize-dequantize in place of a matrix of groups (calibration sweep):
// out = zero + scale * code, one warp per group.
// ---------------------------------------------------------------------------
__global__ void quant_dequant_kernel(int n_groups, const float* __restrict__ x, float clip,
                                     float* __restrict__ out) {
  int gi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gi >= n_groups) return;
  float4 v = reinterpret_cast<const float4*>(x + (size_t)gi * D)[lane];
  float mn = warp_min(fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
  float mx = warp_max(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
  const QParams qp = qparams(mn, mx, clip);
  float4 o;
  o.x = fmaf(qp.s, (float)qcode(v.x, qp), qp.z);
  o.y = fmaf(qp.s, (float)qcode(v.y, qp), qp.z);
  o.z = fmaf(qp.s, (float)qcode(v.z, qp), qp.z);
  o.w = fmaf(qp.s, (float)qcode(v.w, qp), qp.z);
  reinterpret_cast<float4*>(out + (size_t)gi * D)[lane] = o;
}

cudaError_t launch_quant_dequant(int n_groups, const float* x, float clip, float* out,
                                 cudaStream_t s) {
  if (n_groups == 0) return cudaSuccess;
  int blocks = (int)(((long long)n_groups * 32 + 255) / 256);
  quant_dequant_kernel<<<blocks, 256, 0, s>>>(n_groups, x, clip, out);
  return cudaGetLastError();
}

}  // namespace kvq
