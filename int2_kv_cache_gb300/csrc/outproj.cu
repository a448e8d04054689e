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

// y[r][n] = sum_k x[r][k] w[n][k]: a weight-streaming tensor-core GEMM.
//
// With a few activation rows (decode batches) the product is bound by reading W
// once, so the kernel streams W through registers and computes the transposed
// product D[n][r] = W[n][:] . x[r][:] with mma.sync m16n8k16 bf16 -> fp32:
// * A = a 16-row slice of W (row-major, K contiguous): each thread loads 16
//   contiguous bytes of two rows per 32-wide K chunk; the K order inside a
//   chunk is permuted identically in A and B (thread t covers K 8t..8t+7);
// * B = x^T: fp32 activations split into a bf16 high part and a bf16
//   remainder (two MMAs into the same accumulator, ~16 significant bits);
//   fp32 weights are split the same way (three MMAs);
// * a CTA (8 warps) owns 32 rows of W; its warps take K chunks round robin and
//   are summed in shared memory in a fixed order (deterministic).
// grid = ceil(d_model / 32), block = 256; NR = 8-row groups of x per pass (<= 32 rows).
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf_rn(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8 consecutive weights of row n at column k as 4 bf16x2 words (high parts) and,
// for fp32 weights, 4 words of remainders.
template <int WDT>
__device__ __forceinline__ void load_w8(const void* w, size_t off, bool ok, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
  if (!ok) {
    hi[0] = hi[1] = hi[2] = hi[3] = 0u;
    lo[0] = lo[1] = lo[2] = lo[3] = 0u;
    return;
  }
  if (WDT == KVQ_BF16) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(w) + off));
    hi[0] = v.x; hi[1] = v.y; hi[2] = v.z; hi[3] = v.w;
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w) + off));
    const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(w) + off) + 1);
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float h0 = bf_rn(f[2 * i]), h1 = bf_rn(f[2 * i + 1]);
      hi[i] = pack_bf2(h0, h1);
      lo[i] = pack_bf2(f[2 * i] - h0, f[2 * i + 1] - h1);
    }
  }
}

template <int WDT, int NR>
__global__ void __launch_bounds__(256) out_proj_mma_kernel(int n_rows, int d_model, int k_dim,
                                                           const float* __restrict__ x,
                                                           const void* __restrict__ w,
                                                           float* __restrict__ y) {
  __shared__ float red[8][32][8 * NR + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;
  const int n0 = blockIdx.x * 32;
  float acc[2][NR][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;

  const int n_chunks = k_dim / 32;
  for (int ck = warp; ck < n_chunks; ck += 8) {
    const int k = ck * 32 + 8 * ti;
    // B: x rows 8nt+g, columns k..k+7 -> hi/lo bf16 pairs
    uint32_t bx_hi[NR][4], bx_lo[NR][4];
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) {
      const int r = 8 * nt + gi;
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (r < n_rows) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(x + (size_t)r * k_dim + k));
        const float4 b = __ldg(reinterpret_cast<const float4*>(x + (size_t)r * k_dim + k) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float h0 = bf_rn(f[2 * i]), h1 = bf_rn(f[2 * i + 1]);
        bx_hi[nt][i] = pack_bf2(h0, h1);
        bx_lo[nt][i] = pack_bf2(f[2 * i] - h0, f[2 * i + 1] - h1);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int ra = n0 + 16 * mt + gi, rb = ra + 8;
      uint32_t wa_hi[4], wa_lo[4], wb_hi[4], wb_lo[4];
      load_w8<WDT>(w, (size_t)ra * k_dim + k, ra < d_model, wa_hi, wa_lo);
      load_w8<WDT>(w, (size_t)rb * k_dim + k, rb < d_model, wb_hi, wb_lo);
      // two k-steps per 32-wide chunk: step s uses the thread's elements 4s..4s+3
#pragma unroll
      for (int st = 0; st < 2; ++st) {
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          mma_bf16(acc[mt][nt], wa_hi[2 * st], wb_hi[2 * st], wa_hi[2 * st + 1], wb_hi[2 * st + 1],
                   bx_hi[nt][2 * st], bx_hi[nt][2 * st + 1]);
          mma_bf16(acc[mt][nt], wa_hi[2 * st], wb_hi[2 * st], wa_hi[2 * st + 1], wb_hi[2 * st + 1],
                   bx_lo[nt][2 * st], bx_lo[nt][2 * st + 1]);
          if (WDT == KVQ_F32)
            mma_bf16(acc[mt][nt], wa_lo[2 * st], wb_lo[2 * st], wa_lo[2 * st + 1], wb_lo[2 * st + 1],
                     bx_hi[nt][2 * st], bx_hi[nt][2 * st + 1]);
        }
      }
    }
  }
  // D fragment: (row 16mt+g, cols 8nt+2t, +1) and (row 16mt+g+8, same cols)
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) {
      red[warp][16 * mt + gi][8 * nt + 2 * ti] = acc[mt][nt][0];
      red[warp][16 * mt + gi][8 * nt + 2 * ti + 1] = acc[mt][nt][1];
      red[warp][16 * mt + gi + 8][8 * nt + 2 * ti] = acc[mt][nt][2];
      red[warp][16 * mt + gi + 8][8 * nt + 2 * ti + 1] = acc[mt][nt][3];
    }
  __syncthreads();
  for (int e = threadIdx.x; e < 32 * 8 * NR; e += 256) {
    const int nn = e % 32, r = e / 32;
    float v = 0.f;
#pragma unroll
    for (int wv = 0; wv < 8; ++wv) v += red[wv][nn][r];
    if (n0 + nn < d_model && r < n_rows) y[(size_t)r * d_model + n0 + nn] = v;
  }
}

cudaError_t launch_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                            int w_dtype, float* y, cudaStream_t s) {
  if (n_rows == 0 || d_model == 0) return cudaSuccess;
  const dim3 grid((d_model + 31) / 32);
  for (int r0 = 0; r0 < n_rows; r0 += 32) {
    const int nr = n_rows - r0 < 32 ? n_rows - r0 : 32;
    const float* xr = x + (size_t)r0 * k_dim;
    float* yr = y + (size_t)r0 * d_model;
#define KVQ_OP(NRR)                                                                                  \
  if (w_dtype == KVQ_F32) out_proj_mma_kernel<KVQ_F32, NRR><<<grid, 256, 0, s>>>(nr, d_model, k_dim, xr, w, yr); \
  else out_proj_mma_kernel<KVQ_BF16, NRR><<<grid, 256, 0, s>>>(nr, d_model, k_dim, xr, w, yr)
    if (nr <= 8) { KVQ_OP(1); }
    else if (nr <= 16) { KVQ_OP(2); }
    else { KVQ_OP(4); }
#undef KVQ_OP
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvq
