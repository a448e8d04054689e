// W_O folding and the post-W_O output projection.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization", appendix "Equivalent
// Inference Implementation", Eqs. 29-31: W_O-bar_j = W_O,j R_V,h(j), and
// (o_j R_V) W_O-bar_j^T = o_j W_O,j^T; Eq. 3: the layer output sums the heads,
// y = sum_j o_j W_O,j^T = o W_O^T with o the heads concatenated.
#include "quant_common.cuh"

namespace kvq {

// One warp per (row n, query head j): w_folded[n][j] = w[n][j] R_{j / gqa}.
__global__ void fold_wo_kernel(int d_model, int n_q_heads, int gqa, const void* __restrict__ w,
                               int w_dtype, RotDev rot, void* __restrict__ out, int out_dtype) {
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (long long)d_model * n_q_heads) return;
  const int j = (int)(warp % n_q_heads);
  const size_t off = (size_t)warp * D + 4 * lane;
  float4 v = load4(w, off, w_dtype);
  v = rotate_vec_warp(v, rot, j / gqa, lane, false);
  if (out_dtype == KVQ_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + off) = v;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&a);
    pk.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + off) = pk;
  }
}

cudaError_t launch_fold_wo(int d_model, int n_q_heads, int gqa, const void* w, int w_dtype,
                           RotDev rot_v, void* out, int out_dtype, cudaStream_t s) {
  const long long warps = (long long)d_model * n_q_heads;
  if (warps == 0) return cudaSuccess;
  const int blocks = (int)((warps * 32 + 255) / 256);
  fold_wo_kernel<<<blocks, 256, 0, s>>>(d_model, n_q_heads, gqa, w, w_dtype, rot_v, out, out_dtype);
  return cudaGetLastError();
}

// y[r][n] = sum_k x[r][k] w[n][k].  Shared-memory tiled fp32 GEMM:
// block = 256 threads computes a 16 (rows) x 64 (n) tile; each thread 4 outputs.
constexpr int OP_BM = 16, OP_BN = 64, OP_BK = 64;

template <int WDT>
__global__ void __launch_bounds__(256) out_proj_kernel(int n_rows, int d_model, int k_dim,
                                                       const float* __restrict__ x,
                                                       const void* __restrict__ w,
                                                       float* __restrict__ y) {
  __shared__ float xs[OP_BM][OP_BK + 1];
  __shared__ float ws[OP_BN][OP_BK + 1];
  const int r0 = blockIdx.y * OP_BM, n0 = blockIdx.x * OP_BN;
  const int tid = threadIdx.x;
  const int tr = tid / 16;        // row within tile (0..15)
  const int tn = (tid % 16) * 4;  // 4 consecutive n
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < k_dim; k0 += OP_BK) {
    for (int i = tid; i < OP_BM * OP_BK; i += 256) {
      const int rr = i / OP_BK, kk = i % OP_BK;
      const int r = r0 + rr, k = k0 + kk;
      xs[rr][kk] = (r < n_rows && k < k_dim) ? x[(size_t)r * k_dim + k] : 0.f;
    }
    for (int i = tid; i < OP_BN * OP_BK; i += 256) {
      const int nn = i / OP_BK, kk = i % OP_BK;
      const int n = n0 + nn, k = k0 + kk;
      float v = 0.f;
      if (n < d_model && k < k_dim) v = load1(w, (size_t)n * k_dim + k, WDT);
      ws[nn][kk] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < OP_BK; ++kk) {
      const float xv = xs[tr][kk];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = fmaf(xv, ws[tn + i][kk], acc[i]);
    }
    __syncthreads();
  }
  const int r = r0 + tr;
  if (r < n_rows) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (n0 + tn + i < d_model) y[(size_t)r * d_model + n0 + tn + i] = acc[i];
  }
}

cudaError_t launch_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                            int w_dtype, float* y, cudaStream_t s) {
  if (n_rows == 0 || d_model == 0) return cudaSuccess;
  dim3 grid((d_model + OP_BN - 1) / OP_BN, (n_rows + OP_BM - 1) / OP_BM);
  if (w_dtype == KVQ_F32)
    out_proj_kernel<KVQ_F32><<<grid, 256, 0, s>>>(n_rows, d_model, k_dim, x, w, y);
  else
    out_proj_kernel<KVQ_BF16><<<grid, 256, 0, s>>>(n_rows, d_model, k_dim, x, w, y);
  return cudaGetLastError();
}

}  // namespace kvq
