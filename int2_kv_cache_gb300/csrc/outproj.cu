// W_O folding and the post-W_O output projection.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization", appendix "Equivalent
// Inference Implementation", Eqs. 29-31: W_O-bar_j = W_O,j R_V,h(j), and
// (o_j R_V) W_O-bar_j^T = o_j W_O,j^T; Eq. 3: the layer output sums the heads,
// y = sum_j o_j W_O,j^T = o W_O^T with o the heads concatenated.
#include <cuda.h>
#include <cudaTypedefs.h>

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

// bf16 weights, the decode-size case: W streamed once through shared memory by
// the tensor-memory-access engine.
//
// A CTA owns BM = 16 MT rows of W and a pass of up to 8 NR activation rows, and
// is warp-specialised: one producer warp stages each 256-column block of W
// (four 2-D boxes of 64 columns x BM rows) and of x (eight boxes of 32 columns x
// 8 NR rows) into a ring of OP_STAGES shared-memory stages with tensor copies
// (cp.async.bulk.tensor, 128-byte swizzle, out-of-range rows and columns read as
// zeros), and 16 consumer warps each take 16 columns of every stage and release
// it on the stage's "empty" mbarrier - no block barrier in the loop.  The
// swizzle makes the ldmatrix reads of W and the 8-byte reads of x free of bank
// conflicts; x is split into bf16 high and remainder parts (two products into
// one fp32 accumulator); CTAs start at different column blocks (they all share
// x); the consumers' partial sums are added in a fixed order at the end.
constexpr int OP_BK = 256;
constexpr int OP_CW = 16;                   // consumer warps
constexpr int OP_PW = 3;                    // producer warps, 4 tensor copies each per stage
constexpr int OP_THREADS = 32 * (OP_CW + OP_PW);

__host__ __device__ constexpr int op_stage_bytes(int mt, int nr) { return OP_BK * 2 * 16 * mt + OP_BK * 4 * 8 * nr; }
// stages in flight: as many as fit two CTAs per SM (at least 2, at most 4)
__host__ __device__ constexpr int op_stages(int mt, int nr) {
  return (110 * 1024) / op_stage_bytes(mt, nr) >= 4 ? 4 : ((110 * 1024) / op_stage_bytes(mt, nr) >= 2 ? (110 * 1024) / op_stage_bytes(mt, nr) : 2);
}
__host__ __device__ constexpr int op_smem_bytes(int mt, int nr) {
  // stages (1,024-byte aligned for the swizzle) or the final reduction, whichever is larger
  return 1024 + (op_stages(mt, nr) * op_stage_bytes(mt, nr) > OP_CW * 16 * mt * (8 * nr + 1) * 4
                     ? op_stages(mt, nr) * op_stage_bytes(mt, nr)
                     : OP_CW * 16 * mt * (8 * nr + 1) * 4);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

template <int MT, int NR>
__global__ void __launch_bounds__(OP_THREADS) out_proj_tma_kernel(const __grid_constant__ CUtensorMap tw,
                                                                  const __grid_constant__ CUtensorMap tx,
                                                                  int n_rows, int d_model, int k_dim,
                                                                  float* __restrict__ y, unsigned* err) {
  constexpr int BM = 16 * MT, XR = 8 * NR;
  constexpr int WBOX = 128 * BM;          // bytes of one W box (64 bf16 columns x BM rows)
  constexpr int XBOX = 128 * XR;          // bytes of one x box (32 fp32 columns x XR rows)
  constexpr int STAGE = op_stage_bytes(MT, NR);
  constexpr int S = op_stages(MT, NR);
  constexpr int MAX_S = 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[MAX_S], empty[MAX_S];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;
  const int n0 = blockIdx.x * BM;
  const int w_rows = min(BM, d_model - n0);
  const int n_k = (k_dim + OP_BK - 1) / OP_BK;
  const int kc0 = blockIdx.x % n_k;  // CTAs start at different column blocks
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], OP_PW);   // one arrival (with its bytes) per producer warp
      mbar_init(&empty[i], OP_CW);  // one arrival per consumer warp
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp >= OP_CW) {
    // ---- producers: copies q = 4 p + lane (lanes 0-3 of producer p) of the stage's
    //      12 boxes: W boxes 0-3, then x boxes 0-7 ----
    const int q = 4 * (warp - OP_CW) + lane;
    if (warp != OP_CW) pdl_wait();  // x may come from the preceding kernel; W is read before it ends
    int issued = 0;
    for (int kc = 0; kc < n_k; ++kc) {
      const int st = kc % S;
      if (kc >= S) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[st], ((kc / S) - 1) & 1));
        if (!ok || *reinterpret_cast<volatile int*>(&s_abort)) {
          if (!ok && lane == 0) {
            flag_error(err, ERR_TIMEOUT);
            *reinterpret_cast<volatile int*>(&s_abort) = 1;
          }
          break;
        }
      }
      const int k0 = ((kc + kc0) % n_k) * OP_BK;
      uint8_t* dst = smem + st * STAGE;
      if (lane == 0)
        mbar_arrive_expect_tx(&full[st], (uint32_t)(warp == OP_CW ? 4 * WBOX : 4 * XBOX));
      __syncwarp();
      if (lane < 4) {
        if (q < 4) tma_load_2d(dst + q * WBOX, &tw, k0 + 64 * q, n0, &full[st]);
        else tma_load_2d(dst + 4 * WBOX + (q - 4) * XBOX, &tx, k0 + 32 * (q - 4), 0, &full[st]);
      }
      issued = kc + 1;
    }
    // before the CTA retires, wait (bounded) for every stage this warp filled
    for (int kc = (issued > S ? issued - S : 0); kc < issued; ++kc) mbar_wait_bounded(&full[kc % S], (kc / S) & 1);
  }

  float acc[MT][NR][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
  if (warp < OP_CW) {
    // ---- consumers: warp c takes columns 16c .. 16c + 15 of every stage ----
    // W: box c / 4, 16-byte chunks 2 (c % 4) + (lane >> 4) of rows 16 mt + (lane & 15)
    const int wbox = warp >> 2;
    const int wr = (lane & 7) + 8 * ((lane >> 3) & 1);            // row within an m-tile (rows +16 mt keep r % 8)
    const int wch = (2 * (warp & 3) + (lane >> 4)) ^ (wr & 7);    // swizzled chunk
    // x: box c / 2, columns 16 (c % 2) + 2t (+ 8) of rows 8 nt + g
    const int xbox = warp >> 1;
    const int xc0 = 16 * (warp & 1) + 2 * ti;
    const int xch0 = (xc0 >> 2) ^ gi, xch1 = ((xc0 + 8) >> 2) ^ gi;
    const int xoff = (xc0 & 3) * 4;
    for (int kc = 0; kc < n_k; ++kc) {
      const int st = kc % S;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (kc / S) & 1));
      if (!ok || *reinterpret_cast<volatile int*>(&s_abort)) {
        if (!ok && lane == 0) {
          flag_error(err, ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(&s_abort) = 1;
        }
        break;
      }
      const uint8_t* sb = smem + st * STAGE;
      uint32_t a[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        ldsm_x4(smem_u32(sb + wbox * WBOX + (16 * mt + wr) * 128 + wch * 16), a[mt]);
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) {
        const uint8_t* xr = sb + 4 * WBOX + xbox * XBOX + (8 * nt + gi) * 128;
        const float2 p0 = *reinterpret_cast<const float2*>(xr + xch0 * 16 + xoff);
        const float2 p1 = *reinterpret_cast<const float2*>(xr + xch1 * 16 + xoff);
        const float h0 = bf_rn(p0.x), h1 = bf_rn(p0.y), h2 = bf_rn(p1.x), h3 = bf_rn(p1.y);
        const uint32_t bh0 = pack_bf2(h0, h1), bh1 = pack_bf2(h2, h3);
        const uint32_t bl0 = pack_bf2(p0.x - h0, p0.y - h1), bl1 = pack_bf2(p1.x - h2, p1.y - h3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], bh0, bh1);
          mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], bl0, bl1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
  __syncthreads();  // every stage consumed and every copy landed: the stages become the reduction buffer
  pdl_wait();       // y may still be read by the preceding kernel
  if (*reinterpret_cast<volatile int*>(&s_abort)) return;

  // D fragment: (row 16mt+g, cols 8nt+2t, +1) and (row 16mt+g+8, same cols)
  float* red = reinterpret_cast<float*>(smem);  // [OP_CW][BM][XR + 1]
  if (warp < OP_CW) {
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
  }
  __syncthreads();
  for (int e = threadIdx.x; e < BM * XR; e += OP_THREADS) {
    const int nn = e % BM, r = e / BM;
    float v = 0.f;
#pragma unroll
    for (int wv = 0; wv < OP_CW; ++wv) v += red[(wv * BM + nn) * (XR + 1) + r];
    if (nn < w_rows && r < n_rows) y[(size_t)r * d_model + n0 + nn] = v;
  }
}

// Decode-size projection (up to 16 activation rows), split over K in a cluster:
// a cluster of OPC_SPLIT CTAs owns 128 rows of W, CTA r the r-th quarter of the
// columns, so each CTA reads a quarter of x for 128 rows of W.  Stages are 64
// columns wide - one 64 x 128 tensor box of W (16 KB) and two 32-column boxes of
// x - and OPC_STAGES deep (~160 KB in flight per SM).  Consumer warp c takes
// k-step c % 4 (16 columns) of the stage for row tiles 2 (c / 4) and 2 (c / 4) + 1;
// the four k-step warps of a row group are summed in shared memory, then CTA 0
// adds the four partial outputs through distributed shared memory in rank order.
constexpr int OPC_SPLIT = 4;
constexpr int OPC_BM = 128;
constexpr int OPC_BK = 64;
constexpr int OPC_STAGES = 8;

__host__ __device__ constexpr int opc_stage_bytes(int nr) { return OPC_BK * 2 * OPC_BM + OPC_BK * 4 * 8 * nr; }
__host__ __device__ constexpr int opc_red_bytes(int nr) { return 4 * OPC_BM * (8 * nr + 1) * 4; }
__host__ __device__ constexpr int opc_smem_bytes(int nr) {  // stages, or reduction + receive buffers
  return 1024 + (OPC_STAGES * opc_stage_bytes(nr) > opc_red_bytes(nr) + OPC_SPLIT * OPC_BM * 8 * nr * 4
                     ? OPC_STAGES * opc_stage_bytes(nr)
                     : opc_red_bytes(nr) + OPC_SPLIT * OPC_BM * 8 * nr * 4);
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store v at the same shared-memory offset as `local` in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

template <int NR>
__global__ void __launch_bounds__(OP_THREADS) out_proj_cluster_kernel(const __grid_constant__ CUtensorMap tw,
                                                                      const __grid_constant__ CUtensorMap tx,
                                                                      int n_rows, int d_model, int k_dim,
                                                                      float* __restrict__ y, unsigned* err) {
  constexpr int XR = 8 * NR;
  constexpr int WBOX = 128 * OPC_BM;  // 64 bf16 columns x 128 rows
  constexpr int XBOX = 128 * XR;      // 32 fp32 columns x XR rows
  constexpr int STAGE = opc_stage_bytes(NR);
  constexpr int S = OPC_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[S], empty[S];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int n0 = blockIdx.x * OPC_BM;
  const int w_rows = min(OPC_BM, d_model - n0);
  const int n_k_all = (k_dim + OPC_BK - 1) / OPC_BK;
  const int per = (n_k_all + OPC_SPLIT - 1) / OPC_SPLIT;
  const int kc_begin = min(n_k_all, (int)rank * per);
  const int n_k = min(n_k_all, kc_begin + per) - kc_begin;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], OP_CW);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == OP_CW) {
    // ---- producer: lane 0 the W box, lanes 1-2 the x boxes of a stage; the W
    //      boxes of the first stages go out before the preceding kernel ends ----
    int issued = 0;
    bool x_ready = false;
    for (int kc = 0; kc < n_k; ++kc) {
      const int st = kc % S;
      if (kc >= S) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[st], ((kc / S) - 1) & 1));
        if (!ok || *reinterpret_cast<volatile int*>(&s_abort)) {
          if (!ok && lane == 0) {
            flag_error(err, ERR_TIMEOUT);
            *reinterpret_cast<volatile int*>(&s_abort) = 1;
          }
          break;
        }
      }
      const int k0 = (kc_begin + kc) * OPC_BK;
      uint8_t* dst = smem + st * STAGE;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[st], (uint32_t)STAGE);
        tma_load_2d(dst, &tw, k0, n0, &full[st]);
      }
      __syncwarp();  // the byte count is armed before the x copies of this stage
      issued = kc + 1;
      if (kc + 1 == min(n_k, S) || kc >= S) {  // the x boxes of every stage issued so far
        if (!x_ready) {
          pdl_wait();  // x comes from the preceding kernel
          x_ready = true;
        }
        for (int k2 = (kc >= S ? kc : 0); k2 <= kc; ++k2) {
          const int s2 = k2 % S;
          if (lane >= 1 && lane < 3)
            tma_load_2d(smem + s2 * STAGE + WBOX + (lane - 1) * XBOX, &tx, (kc_begin + k2) * OPC_BK + 32 * (lane - 1), 0,
                        &full[s2]);
        }
      }
      __syncwarp();
    }
    if (!x_ready) pdl_wait();
    for (int kc = (issued > S ? issued - S : 0); kc < issued; ++kc) mbar_wait_bounded(&full[kc % S], (kc / S) & 1);
  }

  const int ks = warp & 3, rg = warp >> 2;  // k-step of the stage, row group (tiles 2 rg, 2 rg + 1)
  float acc[2][NR][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NR; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
  if (warp < OP_CW) {
    const int wr = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int wch = (2 * ks + (lane >> 4)) ^ (wr & 7);
    const int xc0 = 16 * (ks & 1) + 2 * ti;  // column within x box ks / 2
    const int xch0 = (xc0 >> 2) ^ gi, xch1 = ((xc0 + 8) >> 2) ^ gi;
    const int xoff = (xc0 & 3) * 4;
    for (int kc = 0; kc < n_k; ++kc) {
      const int st = kc % S;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (kc / S) & 1));
      if (!ok || *reinterpret_cast<volatile int*>(&s_abort)) {
        if (!ok && lane == 0) {
          flag_error(err, ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(&s_abort) = 1;
        }
        break;
      }
      const uint8_t* sb = smem + st * STAGE;
      uint32_t a[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) ldsm_x4(smem_u32(sb + (16 * (2 * rg + mt) + wr) * 128 + wch * 16), a[mt]);
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) {
        const uint8_t* xr = sb + WBOX + (ks >> 1) * XBOX + (8 * nt + gi) * 128;
        const float2 p0 = *reinterpret_cast<const float2*>(xr + xch0 * 16 + xoff);
        const float2 p1 = *reinterpret_cast<const float2*>(xr + xch1 * 16 + xoff);
        const float h0 = bf_rn(p0.x), h1 = bf_rn(p0.y), h2 = bf_rn(p1.x), h3 = bf_rn(p1.y);
        const uint32_t bh0 = pack_bf2(h0, h1), bh1 = pack_bf2(h2, h3);
        const uint32_t bl0 = pack_bf2(p0.x - h0, p0.y - h1), bl1 = pack_bf2(p1.x - h2, p1.y - h3);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], bh0, bh1);
          mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], bl0, bl1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
  __syncthreads();  // every stage consumed and every copy landed
  pdl_wait();       // y may still be read by the preceding kernel
  const bool aborted = *reinterpret_cast<volatile int*>(&s_abort) != 0;
  float* red = reinterpret_cast<float*>(smem);                       // [4 k-steps][128][XR + 1]
  float* recv = reinterpret_cast<float*>(smem + opc_red_bytes(NR));  // [OPC_SPLIT][XR][128] (CTA 0)
  if (warp < OP_CW) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NR; ++nt) {
        float* r0 = red + (ks * OPC_BM + 16 * (2 * rg + mt) + gi) * (XR + 1) + 8 * nt + 2 * ti;
        float* r1 = r0 + 8 * (XR + 1);
        r0[0] = acc[mt][nt][0];
        r0[1] = acc[mt][nt][1];
        r1[0] = acc[mt][nt][2];
        r1[1] = acc[mt][nt][3];
      }
  }
  __syncthreads();
  // every CTA stores its partial into slot `rank` of CTA 0's receive buffer
  for (int e = threadIdx.x; e < OPC_BM * XR; e += OP_THREADS) {
    const int nn = e % OPC_BM, r = e / OPC_BM;
    const float v = ((red[(0 * OPC_BM + nn) * (XR + 1) + r] + red[(1 * OPC_BM + nn) * (XR + 1) + r]) +
                     red[(2 * OPC_BM + nn) * (XR + 1) + r]) + red[(3 * OPC_BM + nn) * (XR + 1) + r];
    st_cluster_f32(recv + rank * OPC_BM * XR + e, 0, v);
  }
  cluster_sync_all();  // release / acquire: every partial has landed in CTA 0
  if (rank == 0 && !aborted) {
    for (int e = threadIdx.x; e < OPC_BM * XR; e += OP_THREADS) {
      const int nn = e % OPC_BM, r = e / OPC_BM;
      float v = recv[e];
#pragma unroll
      for (int q = 1; q < OPC_SPLIT; ++q) v += recv[q * OPC_BM * XR + e];
      if (nn < w_rows && r < n_rows) y[(size_t)r * d_model + n0 + nn] = v;
    }
  }
}

// cuTensorMapEncodeTiled from the driver (no link-time dependency on it).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D row-major [rows][cols] tensor map with 128-byte swizzled boxes of box_cols x box_rows.
static bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base, int rows, int cols,
                      int box_cols, int box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int NR>
cudaError_t launch_out_proj_cluster(int nr, int d_model, int k_dim, const float* x, const void* w, float* y,
                                    unsigned* err, cudaStream_t s) {
  constexpr int smem = opc_smem_bytes(NR);
  static bool attr_set = false;  // one flag per kernel instance
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(out_proj_cluster_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tw, tx;
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, d_model, k_dim, 64, OPC_BM) ||
      !encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, nr, k_dim, 32, 8 * NR))
    return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((d_model + OPC_BM - 1) / OPC_BM, OPC_SPLIT);
  cfg.blockDim = dim3(OP_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = OPC_SPLIT;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, out_proj_cluster_kernel<NR>, tw, tx, nr, d_model, k_dim, y, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MT, int NR>
cudaError_t launch_out_proj_tma(int nr, int d_model, int k_dim, const float* x, const void* w, float* y,
                                unsigned* err, cudaStream_t s) {
  constexpr int smem = op_smem_bytes(MT, NR);
  static bool attr_set = false;  // one flag per kernel instance
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(out_proj_tma_kernel<MT, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tw, tx;
  if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, d_model, k_dim, 64, 16 * MT) ||
      !encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, nr, k_dim, 32, 8 * NR))
    return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((d_model + 16 * MT - 1) / (16 * MT));
  cfg.blockDim = dim3(OP_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, out_proj_tma_kernel<MT, NR>, tw, tx, nr, d_model, k_dim, y, err);
  if (e != cudaSuccess) return e;
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
      if (nr <= 16 && (d_model + OPC_BM - 1) / OPC_BM * OPC_SPLIT >= 100)
        e = nr <= 8 ? launch_out_proj_cluster<1>(nr, d_model, k_dim, xr, w, yr, err, s)
                    : launch_out_proj_cluster<2>(nr, d_model, k_dim, xr, w, yr, err, s);
      else if (nr <= 8) e = wide ? launch_out_proj_tma<2, 1>(nr, d_model, k_dim, xr, w, yr, err, s)
                            : launch_out_proj_tma<1, 1>(nr, d_model, k_dim, xr, w, yr, err, s);
      else if (nr <= 16) e = wide ? launch_out_proj_tma<2, 2>(nr, d_model, k_dim, xr, w, yr, err, s)
                                  : launch_out_proj_tma<1, 2>(nr, d_model, k_dim, xr, w, yr, err, s);
      else e = wide ? launch_out_proj_tma<2, 4>(nr, d_model, k_dim, xr, w, yr, err, s)
                    : launch_out_proj_tma<1, 4>(nr, d_model, k_dim, xr, w, yr, err, s);
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
