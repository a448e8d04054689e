// Calibration sweep: post-W_O NMSE of every candidate rotation x clip ratio.
//
// "Output-aware INT2 KV-cache rotation evaluation" (candidate search on
// calibration queries, selection by the smallest post-W_O NMSE) and
// "Output-Aware Rotation for INT2 KV-Cache Quantization" (Eq. 10: the
// post-W_O attention-output error; appendix calibration details: the
// objective is taken over the final query positions, per KV head).
//
// The squared output error of a head group is evaluated through its Gram
// matrix, which is exact algebra: with W_h = the W_O columns of the query
// heads of KV head h and du = o~ - o (unrotated, concatenated over those heads),
//   ||du W_h^T||^2 = du (W_h^T W_h) du^T.
#include "quant_common.cuh"

namespace kvq {



struct CalibWs {
  float *qf, *qr, *kf, *vf, *xk_hi, *xk_lo, *xv_hi, *xv_lo, *kq, *vq, *o_rot, *o_ref, *o_un, *gram;
};

static size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

static CalibWs carve(void* ws, int n_tok, int n_qpos, int n_kv_heads, int gqa, int joint,
                     size_t* total) {
  const size_t hq = (size_t)n_kv_heads * gqa;
  const size_t qn = (size_t)n_qpos * hq * D, kn = (size_t)n_tok * n_kv_heads * D;
  const size_t gd = joint ? hq * D : (size_t)gqa * D;
  const size_t gn = (joint ? 1 : (size_t)n_kv_heads) * gd * gd;
  const size_t sizes[14] = {qn, qn, kn, kn, kn, kn, kn, kn, kn, kn, qn, qn, qn, gn};
  char* p = static_cast<char*>(ws);
  float* ptrs[14];
  size_t off = 0;
  for (int i = 0; i < 14; ++i) {
    ptrs[i] = reinterpret_cast<float*>(p + off);
    off += align_up(sizes[i] * sizeof(float));
  }
  if (total) *total = off;
  return CalibWs{ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[4], ptrs[5], ptrs[6],
                 ptrs[7], ptrs[8], ptrs[9], ptrs[10], ptrs[11], ptrs[12], ptrs[13]};
}

size_t calib_workspace_bytes(int n_tok, int n_qpos, int n_kv_heads, int gqa, int joint) {
  size_t total = 0;
  carve(nullptr, n_tok, n_qpos, n_kv_heads, gqa, joint, &total);
  return total;
}

// Elementwise conversion to fp32, optionally subtracting a per-(head, channel) mean.
__global__ void to_f32_kernel(size_t n, int n_heads, const void* __restrict__ src, int dtype,
                              const float* __restrict__ mu, float* __restrict__ dst) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float v = load1(src, i, dtype);
  if (mu) v -= mu[i % ((size_t)n_heads * D)];
  dst[i] = v;
}

// Causal attention of the queries at positions n_tok - n_qpos + i against fp32
// keys/values: one block per (query position, query head).
__global__ void __launch_bounds__(128) causal_attn_kernel(int n_tok, int n_qpos, int n_kv_heads,
                                                          int gqa, const float* __restrict__ q,
                                                          const float* __restrict__ k,
                                                          const float* __restrict__ v,
                                                          float* __restrict__ o) {
  extern __shared__ float sc[];  // [n_tok]
  __shared__ __align__(16) float qs[D];
  __shared__ float red[4];
  const int qi = blockIdx.x, j = blockIdx.y, hq = n_kv_heads * gqa, h = j / gqa;
  const int t = n_tok - n_qpos + qi;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  qs[tid] = q[((size_t)qi * hq + j) * D + tid] * INV_SQRT_D;
  __syncthreads();
  float mloc = -INFINITY;
  for (int s = tid; s <= t; s += 128) {
    const float4* kr = reinterpret_cast<const float4*>(k + ((size_t)s * n_kv_heads + h) * D);
    float a = 0.f;
#pragma unroll 8
    for (int c4 = 0; c4 < 32; ++c4) {
      const float4 kk = __ldg(kr + c4);
      const float4 qq = reinterpret_cast<const float4*>(qs)[c4];
      a = fmaf(qq.x, kk.x, a); a = fmaf(qq.y, kk.y, a); a = fmaf(qq.z, kk.z, a); a = fmaf(qq.w, kk.w, a);
    }
    sc[s] = a;
    mloc = fmaxf(mloc, a);
  }
  mloc = warp_max(mloc);
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float sloc = 0.f;
  for (int s = tid; s <= t; s += 128) {
    const float e = __expf(sc[s] - M);
    sc[s] = e;
    sloc += e;
  }
  sloc = warp_sum(sloc);
  if (lane == 0) red[warp] = sloc;
  __syncthreads();
  const float L = red[0] + red[1] + red[2] + red[3];
  float acc = 0.f;
  for (int s = 0; s <= t; ++s) acc = fmaf(sc[s], v[((size_t)s * n_kv_heads + h) * D + tid], acc);
  o[((size_t)qi * hq + j) * D + tid] = acc / L;
}

// Gram matrices G_g = W_g^T W_g for head groups g of gd = cols columns each.
// w: [d_model][n_groups * gd]; gram: [n_groups][gd][gd].  32x32 tiles.
__global__ void __launch_bounds__(256) gram_kernel(int d_model, int total_cols, int gd,
                                                   const void* __restrict__ w, int w_dtype,
                                                   float* __restrict__ gram) {
  __shared__ float A[32][33], B[32][33];
  const int grp = blockIdx.z;
  const int a0 = blockIdx.y * 32, b0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // ty 0..7
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const size_t col0 = (size_t)grp * gd;
  for (int n0 = 0; n0 < d_model; n0 += 32) {
    for (int i = ty; i < 32; i += 8) {
      const int n = n0 + i;
      A[i][tx] = n < d_model ? load1(w, (size_t)n * total_cols + col0 + a0 + tx, w_dtype) : 0.f;
      B[i][tx] = n < d_model ? load1(w, (size_t)n * total_cols + col0 + b0 + tx, w_dtype) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int i = 0; i < 32; ++i) {
      const float bv = B[i][tx];
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[r] = fmaf(A[i][ty + 8 * r], bv, acc[r]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
    gram[((size_t)grp * gd + a0 + ty + 8 * r) * gd + b0 + tx] = acc[r];
}

// out[slot] += sum over (position, group) of du G du^T with du = (a - b) (or a when b == NULL).
// grid = (n_qpos, n_groups), block = 256.
__global__ void __launch_bounds__(256) gram_form_kernel(int n_qpos, int n_groups, int gd,
                                                        const float* __restrict__ a,
                                                        const float* __restrict__ b,
                                                        const float* __restrict__ gram,
                                                        double* __restrict__ out) {
  extern __shared__ float du[];  // [gd]
  __shared__ float red[8];
  const int qi = blockIdx.x, grp = blockIdx.y, tid = threadIdx.x;
  const size_t base = ((size_t)qi * n_groups + grp) * gd;
  for (int i = tid; i < gd; i += 256) du[i] = b ? a[base + i] - b[base + i] : a[base + i];
  __syncthreads();
  const float* G = gram + (size_t)grp * gd * gd;
  float part = 0.f;
  for (int c = tid; c < gd; c += 256) {
    float wsum = 0.f;
    for (int r = 0; r < gd; ++r) wsum = fmaf(G[(size_t)r * gd + c], du[r], wsum);
    part = fmaf(wsum, du[c], part);
  }
  part = warp_sum(part);
  if ((tid & 31) == 0) red[tid >> 5] = part;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int i = 0; i < 8; ++i) s += (double)red[i];
    atomicAdd(out + grp, s);
  }
}

// out[slot] += sum over (position, group) of ||du W_g^T||^2 computed directly
// (used when d_model <= the group width, where it is also the cheaper form).
// One warp per output row n of W; grid = (n_qpos, n_groups), block = 256.
__global__ void __launch_bounds__(256) proj_err_kernel(int n_qpos, int n_groups, int gd, int d_model,
                                                       const float* __restrict__ a,
                                                       const float* __restrict__ b,
                                                       const void* __restrict__ w, int w_dtype,
                                                       double* __restrict__ out) {
  extern __shared__ float du[];  // [gd]
  __shared__ double red[8];
  const int qi = blockIdx.x, grp = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t base = ((size_t)qi * n_groups + grp) * gd;
  for (int i = tid; i < gd; i += 256) du[i] = b ? a[base + i] - b[base + i] : a[base + i];
  __syncthreads();
  const size_t total_cols = (size_t)n_groups * gd, col0 = (size_t)grp * gd;
  double part = 0.0;
  for (int n = warp; n < d_model; n += 8) {
    float y = 0.f;
    for (int k = lane; k < gd; k += 32) y = fmaf(du[k], load1(w, (size_t)n * total_cols + col0 + k, w_dtype), y);
    y = warp_sum(y);
    part += (double)y * (double)y;
  }
  if (lane == 0) red[warp] = part;
  __syncthreads();
  if (tid == 0) {
    double s2 = 0.0;
    for (int i = 0; i < 8; ++i) s2 += red[i];
    atomicAdd(out + grp, s2);
  }
}

__global__ void zero_f64_kernel(double* p, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0.0;
}

__global__ void divide_kernel(double* nmse, const double* ref, int n, int n_groups) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) nmse[i] = nmse[i] / ref[i % n_groups];
}

#define KVQ_TRY(x)                          \
  do {                                      \
    cudaError_t e_ = (x);                   \
    if (e_ != cudaSuccess) return e_;       \
    e_ = cudaGetLastError();                \
    if (e_ != cudaSuccess) return e_;       \
  } while (0)

cudaError_t launch_calib(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model,
                         const void* q, const void* k, const void* v, int dtype, const void* w_o,
                         int w_dtype, int n_cand, const kvq_rot* cand, int n_clip,
                         const float* clips, const float* mu, int joint, double* nmse,
                         double* ref, void* ws, cudaStream_t s) {
  const int hq = n_kv_heads * gqa;
  const int n_groups = joint ? 1 : n_kv_heads;
  const int gd = joint ? hq * D : gqa * D;
  CalibWs w = carve(ws, n_tok, n_qpos, n_kv_heads, gqa, joint, nullptr);
  const size_t qn = (size_t)n_qpos * hq * D, kn = (size_t)n_tok * n_kv_heads * D;
  auto blocks = [](size_t n) { return (unsigned)((n + 255) / 256); };

  to_f32_kernel<<<blocks(qn), 256, 0, s>>>(qn, hq, q, dtype, nullptr, w.qf);
  to_f32_kernel<<<blocks(kn), 256, 0, s>>>(kn, n_kv_heads, k, dtype, nullptr, w.kf);
  to_f32_kernel<<<blocks(kn), 256, 0, s>>>(kn, n_kv_heads, v, dtype, nullptr, w.vf);
  KVQ_TRY(cudaSuccess);
  const size_t attn_smem = (size_t)n_tok * sizeof(float);
  // reference readout with unquantized, unrotated, uncentred keys and values
  causal_attn_kernel<<<dim3(n_qpos, hq), 128, attn_smem, s>>>(n_tok, n_qpos, n_kv_heads, gqa, w.qf,
                                                              w.kf, w.vf, w.o_ref);
  KVQ_TRY(cudaSuccess);
  // ||du W^T||^2: directly when d_model <= gd, else through the group's Gram matrix
  const bool direct = d_model <= gd;
  if (!direct)
    gram_kernel<<<dim3(gd / 32, gd / 32, n_groups), 256, 0, s>>>(d_model, hq * D, gd, w_o, w_dtype, w.gram);
  zero_f64_kernel<<<1, 256, 0, s>>>(ref, n_groups);
  const int n_out = n_cand * n_clip * n_groups;
  zero_f64_kernel<<<(n_out + 255) / 256, 256, 0, s>>>(nmse, n_out);
  KVQ_TRY(cudaSuccess);
  const size_t form_smem = (size_t)gd * sizeof(float);
  auto out_err = [&](const float* a, const float* b, double* dst) {
    if (direct)
      proj_err_kernel<<<dim3(n_qpos, n_groups), 256, form_smem, s>>>(n_qpos, n_groups, gd, d_model, a, b, w_o,
                                                                     w_dtype, dst);
    else
      gram_form_kernel<<<dim3(n_qpos, n_groups), 256, form_smem, s>>>(n_qpos, n_groups, gd, a, b, w.gram, dst);
  };
  out_err(w.o_ref, nullptr, ref);
  KVQ_TRY(cudaSuccess);
  for (int i = 0; i < n_cand; ++i) {
    const RotDev r = to_dev(cand[i]);
    // keys centred (OptR §4.1; attention-equivalent) then rotated; values rotated
    KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, k, dtype, mu, r, w.xk_hi, w.xk_lo, s));
    KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, v, dtype, nullptr, r, w.xv_hi, w.xv_lo, s));
    KVQ_TRY(launch_rotate_heads(n_qpos, hq, gqa, w.qf, r, w.qr, false, s));
    for (int c = 0; c < n_clip; ++c) {
      KVQ_TRY(launch_quant_dequant(n_tok * n_kv_heads, w.xk_hi, w.xk_lo, clips[c], w.kq, s));
      KVQ_TRY(launch_quant_dequant(n_tok * n_kv_heads, w.xv_hi, w.xv_lo, clips[c], w.vq, s));
      causal_attn_kernel<<<dim3(n_qpos, hq), 128, attn_smem, s>>>(n_tok, n_qpos, n_kv_heads, gqa,
                                                                  w.qr, w.kq, w.vq, w.o_rot);
      KVQ_TRY(cudaSuccess);
      KVQ_TRY(launch_rotate_heads(n_qpos, hq, gqa, w.o_rot, r, w.o_un, true, s));
      double* slot = nmse + (size_t)(i * n_clip + c) * n_groups;
      out_err(w.o_un, w.o_ref, slot);
      KVQ_TRY(cudaSuccess);
    }
  }
  divide_kernel<<<(n_out + 255) / 256, 256, 0, s>>>(nmse, ref, n_out, n_groups);
  return cudaGetLastError();
}

}  // namespace kvq
