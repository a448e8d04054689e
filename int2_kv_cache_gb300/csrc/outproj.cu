// W_O folding and the post-W_O output projection.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization", appendix "Equivalent
// Inference Implementation", Eqs. 29-31: W_O-bar_j = W_O,j R_V,h(j), and
// (o_j R_V) W_O-bar_j^T = o_j W_O,j^T; Eq. 3: the layer output sums the heads,
// y = sum_j o_j W_O,j^T = o W_O^T with o the heads concatenated.
#include "async_copy.cuh"
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

// bf16 weights, the decode-size case: W streamed through shared memory.
//
// A CTA owns BM = 16 MT rows of W and a pass of up to 8 NR activation rows.
// W (row slices of BK columns) and the matching x columns are staged in a
// ring of shared-memory stages by bulk copies (one row per lane, completed on
// an mbarrier), so tens of kilobytes per SM are in flight; rows are padded by
// 16 (W) and 32 (x) bytes so the ldmatrix reads of W and the 8-byte reads of
// x are free of bank conflicts.  Warp w takes columns BK/8 w .. BK/8 (w + 1) - 1 of every stage; x is
// split into bf16 high and remainder parts (two products into one fp32
// accumulator); the eight warps are summed in a fixed order at the end.
constexpr int OP_MAX_STAGES = 4;
constexpr int OP_SMEM_TARGET = 110 * 1024;  // two CTAs per SM

__host__ __device__ constexpr int op_stage_bytes(int mt, int nr, int bk) {
  return 16 * mt * (bk * 2 + 16) + 8 * nr * (bk * 4 + 32);
}
__host__ __device__ constexpr int op_stages(int mt, int nr, int bk) {
  return OP_SMEM_TARGET / op_stage_bytes(mt, nr, bk) > OP_MAX_STAGES ? OP_MAX_STAGES
         : OP_SMEM_TARGET / op_stage_bytes(mt, nr, bk) < 2          ? 2
                                                                      : OP_SMEM_TARGET / op_stage_bytes(mt, nr, bk);
}

// BK = 256 for up to 32 activation rows, 128 for 64 (so two CTAs still fit an SM).
template <int MT, int NR, int BK>
__global__ void __launch_bounds__(256) out_proj_stream_kernel(int n_rows, int d_model, int k_dim,
                                                              const float* __restrict__ x,
                                                              const __nv_bfloat16* __restrict__ w,
                                                              float* __restrict__ y, unsigned* err) {
  constexpr int BM = 16 * MT, XR = 8 * NR;
  constexpr int KS = BK / 128;        // 16-wide k-steps per warp per stage
  constexpr int WROW = BK * 2 + 16;   // bytes per staged W row
  constexpr int XROW = BK * 4 + 32;   // bytes per staged x row
  constexpr int STAGE = op_stage_bytes(MT, NR, BK);
  constexpr int S = op_stages(MT, NR, BK);
  static_assert(BM <= 32 && XR <= 64, "row-to-thread mapping of the copies");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[OP_MAX_STAGES];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;
  const int n0 = blockIdx.x * BM;
  const int w_rows = min(BM, d_model - n0);
  const int n_k = (k_dim + BK - 1) / BK;

  // One arrival per row copy: every copying thread arms the barrier with its own
  // bytes, so the copies need no ordering among threads.
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&full[i], (uint32_t)(w_rows + n_rows));
    fence_mbar_init();
  }
  __syncthreads();

  // CTAs start at different column blocks, so at any moment they read different
  // slices of x (all of them share x).
  const int kc0 = blockIdx.x % n_k;
  // The row this thread stages: W row `lane * 8 + warp` for lanes 0..3 of each
  // warp (BM <= 32), x row `(lane - 4) * 8 + warp` for lanes 4..11 (<= 64 rows),
  // so the copies of a stage are spread over all eight warps.
  const int my_wr = lane < 4 ? lane * 8 + warp : -1;
  const int my_xr = (lane >= 4 && lane < 12) ? (lane - 4) * 8 + warp : -1;
  const bool copies_w = my_wr >= 0 && my_wr < w_rows;
  const bool copies_x = my_xr >= 0 && my_xr < n_rows;
  auto issue = [&](int kc) {
    if (!copies_w && !copies_x) return;
    const int st = kc % S;
    const int k0 = ((kc + kc0) % n_k) * BK;
    const int kw = min(BK, k_dim - k0);
    uint8_t* dst = smem + st * STAGE;
    fence_proxy_async();
    if (copies_w) {
      mbar_arrive_expect_tx(&full[st], (uint32_t)kw * 2);
      bulk_g2s(dst + my_wr * WROW, w + (size_t)(n0 + my_wr) * k_dim + k0, (uint32_t)kw * 2, &full[st]);
    } else {
      mbar_arrive_expect_tx(&full[st], (uint32_t)kw * 4);
      bulk_g2s(dst + BM * WROW + my_xr * XROW, x + (size_t)my_xr * k_dim + k0, (uint32_t)kw * 4, &full[st]);
    }
  };
  for (int kc = 0; kc < S && kc < n_k; ++kc) issue(kc);

  float acc[MT][NR][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
  // ldmatrix row of this lane: matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15) of an m-tile
  const uint32_t a_off = ((lane & 7) + 8 * ((lane >> 3) & 1)) * WROW + 16 * (lane >> 4);

  for (int kc = 0; kc < n_k; ++kc) {
    const int st = kc % S;
    const bool ok = mbar_wait_bounded(&full[st], (kc / S) & 1);
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) flag_error(err, ERR_TIMEOUT);
      // wait (bounded) for the copies in flight before the CTA retires
      for (int k2 = kc; k2 < n_k && k2 < kc + S; ++k2) mbar_wait_bounded(&full[k2 % S], (k2 / S) & 1);
      return;
    }
    const int kw = min(BK, k_dim - ((kc + kc0) % n_k) * BK);
    if (BK / 8 * warp < kw) {
      const uint8_t* sb = smem + st * STAGE;
      const uint32_t sa = smem_u32(sb) + a_off;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int kb = BK / 8 * warp + 16 * ks;
        uint32_t a[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) ldsm_x4(sa + 16 * mt * WROW + kb * 2, a[mt]);
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
          const float* xr = reinterpret_cast<const float*>(sb + BM * WROW + (8 * nt + gi) * XROW) + kb + 2 * ti;
          const float2 p0 = *reinterpret_cast<const float2*>(xr);
          const float2 p1 = *reinterpret_cast<const float2*>(xr + 8);
          const float h0 = bf_rn(p0.x), h1 = bf_rn(p0.y), h2 = bf_rn(p1.x), h3 = bf_rn(p1.y);
          const uint32_t bh0 = pack_bf2(h0, h1), bh1 = pack_bf2(h2, h3);
          const uint32_t bl0 = pack_bf2(p0.x - h0, p0.y - h1), bl1 = pack_bf2(p1.x - h2, p1.y - h3);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], bh0, bh1);
            mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], bl0, bl1);
          }
        }
      }
    }
    __syncthreads();  // stage st consumed by every warp
    if (kc + S < n_k) issue(kc + S);
  }

  // D fragment: (row 16mt+g, cols 8nt+2t, +1) and (row 16mt+g+8, same cols)
  float* red = reinterpret_cast<float*>(smem);  // [8][BM][XR + 1]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) {
      float* r0 = red + (warp * BM + 16 * mt + gi) * (XR + 1) + 8 * nt + 2 * ti;
      float* r1 = r0 + 8 * (XR + 1);
      r0[0] = acc[mt][nt][0];
      r0[1] = acc[mt][nt][1];
      r1[0] = acc[mt][nt][2];
      r1[1] = acc[mt][nt][3];
    }
  __syncthreads();
  for (int e = threadIdx.x; e < BM * XR; e += 256) {
    const int nn = e % BM, r = e / BM;
    float v = 0.f;
#pragma unroll
    for (int wv = 0; wv < 8; ++wv) v += red[(wv * BM + nn) * (XR + 1) + r];
    if (nn < w_rows && r < n_rows) y[(size_t)r * d_model + n0 + nn] = v;
  }
}

template <int MT, int NR, int BK>
cudaError_t launch_out_proj_stream(int nr, int d_model, int k_dim, const float* x, const void* w, float* y,
                                   unsigned* err, cudaStream_t s) {
  constexpr int smem = op_stages(MT, NR, BK) * op_stage_bytes(MT, NR, BK);
  static_assert(smem >= 8 * 16 * MT * (8 * NR + 1) * 4, "the final reduction reuses the stages");
  static bool attr_set = false;  // one flag per kernel instance
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(out_proj_stream_kernel<MT, NR, BK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = (d_model + 16 * MT - 1) / (16 * MT);
  out_proj_stream_kernel<MT, NR, BK><<<grid, 256, smem, s>>>(nr, d_model, k_dim, x,
                                                              static_cast<const __nv_bfloat16*>(w), y, err);
  return cudaGetLastError();
}

cudaError_t launch_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                            int w_dtype, float* y, unsigned* err, cudaStream_t s) {
  if (n_rows == 0 || d_model == 0) return cudaSuccess;
  const dim3 grid((d_model + 31) / 32);
  const int pass_rows = 32;  // one pass per 32 activation rows (a 64-row pass measured slower)
  for (int r0 = 0; r0 < n_rows; r0 += pass_rows) {
    const int nr = n_rows - r0 < pass_rows ? n_rows - r0 : pass_rows;
    const float* xr = x + (size_t)r0 * k_dim;
    float* yr = y + (size_t)r0 * d_model;
    if (w_dtype == KVQ_BF16) {
      // 32-row W blocks when they alone give ~a CTA per SM, else 16-row blocks
      const bool wide = (d_model + 31) / 32 >= 100;
      cudaError_t e;
      if (nr <= 8) e = wide ? launch_out_proj_stream<2, 1, 256>(nr, d_model, k_dim, xr, w, yr, err, s)
                            : launch_out_proj_stream<1, 1, 256>(nr, d_model, k_dim, xr, w, yr, err, s);
      else if (nr <= 16) e = wide ? launch_out_proj_stream<2, 2, 256>(nr, d_model, k_dim, xr, w, yr, err, s)
                                  : launch_out_proj_stream<1, 2, 256>(nr, d_model, k_dim, xr, w, yr, err, s);
      else if (nr <= 32) e = wide ? launch_out_proj_stream<2, 4, 256>(nr, d_model, k_dim, xr, w, yr, err, s)
                                  : launch_out_proj_stream<1, 4, 256>(nr, d_model, k_dim, xr, w, yr, err, s);
      else e = wide ? launch_out_proj_stream<2, 8, 128>(nr, d_model, k_dim, xr, w, yr, err, s)
                    : launch_out_proj_stream<1, 8, 128>(nr, d_model, k_dim, xr, w, yr, err, s);
      if (e != cudaSuccess) return e;
      continue;
    }
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
