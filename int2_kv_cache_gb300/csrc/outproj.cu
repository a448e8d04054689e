// W_O folding and the post-W_O output projection.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization", appendix "Equivalent
// Inference Implementation", Eqs. 29-31: W_O-bar_j = W_O,j R_V,h(j), and
// (o_j R_V) W_O-bar_j^T = o_j W_O,j^T; Eq. 3: the layer output sums the heads,
// y = sum_j o_j W_O,j^T = o W_O^T with o the heads concatenated.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "async_copy.cuh"
#include "quant_common.cuh"
#include "tcgen05.cuh"

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

// y[r][n] = sum_k x[r][k] w[n][k]: weight-streaming tensor-core GEMMs.  With a
// few activation rows (decode batches) the product is bound by reading W once.
//
// fp32 weights: the kernel streams W through registers and computes the transposed
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

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// bf16 weights on the fifth-generation tensor cores (tcgen05), split over K in
// a cluster.  D[n][c] = sum_k W[n][k] B[c][k] with M = 128 rows of W per CTA
// and N = 2 NRP columns: B holds the pass's activation rows twice, as bf16
// high parts (columns 0 .. NRP-1) and bf16 remainders (NRP .. 2 NRP-1), so
// y[r][n] = D[n][r] + D[n][NRP + r] keeps ~16 bits of x against bf16 W.
// K advances in 64-column stages through three shared-memory rings sized
// independently - W (read from memory once), x (read by every row tile, from
// L2) and the converted B tiles:
// * warp 0 streams the 128 x 64 boxes of W into a ring of SW stages by tensor
//   copies (128-byte swizzle, zero fill past the edges);
// * warps 4-11 fetch x (fp32) with per-thread asynchronous copies into a ring of
//   SX stages, once the preceding kernel (which writes x) has finished, split
//   each stage into the bf16 B tile (128-byte swizzle) in a ring of SB stages
//   and release it to the tensor core;
// * one thread of warp 1 issues four 128 x N x 16 MMAs per stage into tensor
//   memory, then commits them to the W stage's and the B stage's "free" barriers;
// * warps 4-7 read the accumulator back (warp w: lanes 32 (w % 4) ..), and the
//   cluster's K partials meet by distributed shared memory: rank j receives
//   rows [j rpr, (j + 1) rpr) of every CTA's tile and adds them in rank order.
// Every wait is bounded (error flag and early exit; the cluster barriers are
// always reached); tensor memory is freed by the warp that took it.
constexpr int OPT_BM = 128;
constexpr int OPT_BK = 64;
constexpr int OPT_THREADS = 384;
constexpr int OPT_WBYTES = OPT_BM * 128;  // one W stage: 128 rows x 64 bf16

__host__ __device__ constexpr int opt_xbytes(int nrp) { return 256 * nrp; }  // x stage: NRP rows x 64 fp32
__host__ __device__ constexpr int opt_bbytes(int nrp) { return 256 * nrp; }  // B stage: 2 NRP rows x 64 bf16
// x and B ring depths: the x copies (from L2) and the B round trip (convert,
// MMA, commit) each take about a microsecond.  Up to 16 activation rows two CTAs
// share an SM (97 KB of rings each, <= 84 registers), with twice the K split:
// 16 x 4096 x 4096 measured 11.6 us against 13.7 us with one CTA per SM.
__host__ __device__ constexpr int opt_ctas_per_sm(int nrp) { return nrp <= 16 ? 2 : 1; }
__host__ __device__ constexpr int opt_sx(int nrp) { return nrp <= 16 ? 4 : (nrp <= 32 ? 6 : 4); }
__host__ __device__ constexpr int opt_sb(int nrp) { return nrp <= 16 ? 4 : (nrp <= 32 ? 6 : 4); }
// W ring depth: four 16 KB boxes in flight per SM measured fastest (deeper rings
// of these 128-row boxes lost up to 40% on GB300)
__host__ __device__ constexpr int opt_sw(int) { return 4; }
__host__ __device__ constexpr int opt_smem_bytes(int nrp) {
  return 1024 + opt_sw(nrp) * OPT_WBYTES + opt_sx(nrp) * opt_xbytes(nrp) + opt_sb(nrp) * opt_bbytes(nrp);
}

// x -> (hi, lo) bf16 pairs of two values: hi = bf16(x) rounded to nearest even,
// lo = bf16(x - hi); hi + lo keeps ~16 significant bits of x.
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf2(a, b);
  lo = pack_bf2(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}

// 16-byte global -> shared copy through L2 (cp.async, completion by commit groups).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory address of `local_base` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* local_base, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_base)), "r"(rank));
  return remote;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// PACKED: W comes pre-tiled (kvq_pack_wo): the box of row tile T and K stage c is the
// contiguous 16 KB at (T n_kb + c) * 16 KB, already in the shared-memory order a 128-byte
// swizzled tensor copy would produce, so one bulk copy moves it (one DRAM stream per box
// instead of 128 rows of 128 bytes).
template <int NRP, bool PACKED>
__global__ void __launch_bounds__(OPT_THREADS, opt_ctas_per_sm(NRP)) out_proj_tc_kernel(const __grid_constant__ CUtensorMap tw,
                                                                     const uint8_t* __restrict__ wpack,
                                                                     const float* __restrict__ x, int n_rows,
                                                                     int d_model, int k_dim, float* __restrict__ y,
                                                                     unsigned* err) {
  constexpr int N = 2 * NRP;
  constexpr int SW = opt_sw(NRP), SX = opt_sx(NRP), SB = opt_sb(NRP);
  constexpr int XS = opt_xbytes(NRP), BS = opt_bbytes(NRP);
  constexpr uint32_t TCOLS = N < 32 ? 32 : N;
  constexpr uint32_t IDESC = idesc_bf16_f32(OPT_BM, N);
  constexpr unsigned FULLM = 0xffffffffu;
  static_assert(N >= 16 && N <= 256 && N % 16 == 0, "tcgen05 M=128 tile needs 16 <= N <= 256, N % 16 == 0");
  static_assert(XS % 1024 == 0 && BS % 1024 == 0, "ring stages stay 1,024-byte aligned (128-byte swizzle)");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* xring = smem + SW * OPT_WBYTES;
  uint8_t* bring = xring + SX * XS;
  __shared__ __align__(8) uint64_t wfull[SW], wfree[SW], bfull[SB], bfree[SB];
  __shared__ __align__(8) uint64_t adone;  // one phase: every MMA of the CTA has completed
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t rank, split;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(split));
  const int n0 = blockIdx.x * OPT_BM;
  const int n_kb = (k_dim + OPT_BK - 1) / OPT_BK;
  const int kb0 = (int)((long long)n_kb * rank / split);
  const int n_k = (int)((long long)n_kb * (rank + 1) / split) - kb0;  // >= 1: split <= n_kb
  if (threadIdx.x == 0) {
    for (int i = 0; i < SW; ++i) {
      mbar_init(&wfull[i], 1);  // the W producer's arrival (with the box's bytes)
      mbar_init(&wfree[i], 1);  // the MMA commit
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bfull[i], OPT_THREADS / 32 - 4);  // one arrival per converter warp
      mbar_init(&bfree[i], 1);  // the MMA commit
    }
    mbar_init(&adone, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };
  auto give_up = [&]() {
    flag_error(err, ERR_TIMEOUT);
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
  };
  // bounded, warp-uniform wait; false (and the CTA marked aborted) on a time-out
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    const bool ok = __all_sync(FULLM, mbar_wait_bounded(bar, parity));
    if (!ok && lane == 0) give_up();
    return ok && !aborted();
  };

  if (warp == 0) {
    // ---- W producer ----
    // A row-major W may come from the preceding kernel (a fold right before the
    // projection): wait for it.  A packed W is static (written before the preceding
    // kernel began): stream it while that kernel still runs.
    if (!PACKED) pdl_wait();
    int issued = 0;
    for (int kb = 0; kb < n_k; ++kb) {
      const int st = kb % SW;
      if (kb >= SW && !warp_wait(&wfree[st], ((kb / SW) - 1) & 1)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&wfull[st], OPT_WBYTES);
        if (PACKED)
          bulk_g2s(wring + st * OPT_WBYTES, wpack + ((size_t)blockIdx.x * n_kb + kb0 + kb) * OPT_WBYTES, OPT_WBYTES,
                   &wfull[st]);
        else
          tma_load_2d(wring + st * OPT_WBYTES, &tw, (kb0 + kb) * OPT_BK, n0, &wfull[st]);
      }
      __syncwarp();
      issued = kb + 1;
    }
    // every copy has landed before the ring is reused or the CTA retires
    for (int kb = (issued > SW ? issued - SW : 0); kb < issued; ++kb)
      mbar_wait_bounded(&wfull[kb % SW], (kb / SW) & 1);
  } else if (warp == 1) {
    // ---- MMA issue ----
    int last = -1;
    for (int kb = 0; kb < n_k; ++kb) {
      const int sw = kb % SW, sb = kb % SB;
      if (!warp_wait(&wfull[sw], (kb / SW) & 1)) break;
      if (!warp_wait(&bfull[sb], (kb / SB) & 1)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t ad = sw128_desc(wring + sw * OPT_WBYTES), bd = sw128_desc(bring + sb * BS);
#pragma unroll
        for (int kk = 0; kk < OPT_BK / 16; ++kk) tc_mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, IDESC, kb > 0 || kk > 0);
        tc_commit(&wfree[sw]);
        tc_commit(&bfree[sb]);
      }
      __syncwarp();
      last = kb;
    }
    // the accumulator is complete (or the loop was abandoned) once every MMA
    // issued has completed: no tensor-core work in flight past this point
    if (lane == 0 && last >= 0) tc_commit(&adone);
    __syncwarp();
    if (last >= 0) mbar_wait_bounded(&adone, 0);
  } else if (warp >= 4) {
    // ---- x -> bf16 high / remainder B tile (warps 4-11) ----
    // Thread ct owns items i = ct + 256 t (row i / 8, columns 8 (i % 8) .. + 7 of
    // the stage): it copies their x into its own slots of the x ring with
    // cp.async (SX - 1 stages ahead) and converts them, so x needs no barrier.
    constexpr int CT = OPT_THREADS - 128;          // converter threads
    constexpr int IT = (NRP * 8 + CT - 1) / CT;   // items per thread and stage
    const int ct = threadIdx.x - 128;
    pdl_wait();  // x comes from the preceding kernel
    auto fetch = [&](int kb) {  // stage kb's items -> x ring slot kb % SX (one commit group)
      if (kb < n_k) {
        uint8_t* xs = xring + (kb % SX) * XS;
        const int k0 = (kb0 + kb) * OPT_BK;
#pragma unroll
        for (int t = 0; t < IT; ++t) {
          const int i = ct + CT * t;
          const int r = i >> 3, col = k0 + 8 * (i & 7);
          if (i < NRP * 8 && r < n_rows && col < k_dim) {
            const float* src = x + (size_t)r * k_dim + col;
            cp_async16(xs + i * 32, src);
            cp_async16(xs + i * 32 + 16, src + 4);
          }
        }
      }
      cp_async_commit();
    };
    for (int kb = 0; kb < SX - 1; ++kb) fetch(kb);
    for (int kb = 0; kb < n_k; ++kb) {
      const int sb = kb % SB;
      fetch(kb + SX - 1);  // into the slot converted in the previous iteration
      cp_async_wait<SX - 1>();  // this thread's copies of stage kb have landed
      if (kb >= SB && !warp_wait(&bfree[sb], ((kb / SB) - 1) & 1)) break;
      const uint8_t* xs = xring + (kb % SX) * XS;
      uint8_t* bs = bring + sb * BS;
      const int k0 = (kb0 + kb) * OPT_BK;
      // all of the thread's x first (independent loads), then the B stores
      float4 xa[IT], xb[IT];
#pragma unroll
      for (int t = 0; t < IT; ++t) {
        const int i = ct + CT * t;
        xa[t] = xb[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < NRP * 8 && (i >> 3) < n_rows && k0 + 8 * (i & 7) < k_dim) {
          xa[t] = *reinterpret_cast<const float4*>(xs + i * 32);
          xb[t] = *reinterpret_cast<const float4*>(xs + i * 32 + 16);
        }
      }
#pragma unroll
      for (int t = 0; t < IT; ++t) {
        const int i = ct + CT * t;
        if (i < NRP * 8) {
          const int r = i >> 3, j = i & 7, sw = r & 7;  // row, 16-byte chunk (8 columns) of the B row
          uint4 hi, lo;
          split_bf2(xa[t].x, xa[t].y, hi.x, lo.x);
          split_bf2(xa[t].z, xa[t].w, hi.y, lo.y);
          split_bf2(xb[t].x, xb[t].y, hi.z, lo.z);
          split_bf2(xb[t].z, xb[t].w, hi.w, lo.w);
          *reinterpret_cast<uint4*>(bs + r * 128 + (j ^ sw) * 16) = hi;
          *reinterpret_cast<uint4*>(bs + (NRP + r) * 128 + (j ^ sw) * 16) = lo;
        }
      }
      fence_proxy_async();  // the tensor cores read B through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&bfull[sb]);
    }
    cp_async_wait<0>();  // no copy in flight when the ring is reused
  }

  // ---- epilogue: accumulator rows -> registers (warps 4-7) ----
  const int q4 = warp & 3;
  const int m = 32 * q4 + lane;  // row of the W tile held by this thread
  float v[NRP];
#pragma unroll
  for (int i = 0; i < NRP; ++i) v[i] = 0.f;
  if (warp >= 4 && warp < 8) {
    bool ok = !aborted();
    // a separate one-phase barrier: the stage barriers' parities cannot tell how
    // many rounds behind the tensor core is
    if (ok) ok = mbar_wait_bounded(&adone, 0);
    ok = __all_sync(FULLM, ok);
    if (!ok && lane == 0 && !aborted()) give_up();
    tc_fence_after();
    if (ok) {
      const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
#pragma unroll
      for (int c = 0; c < NRP; c += 8) {
        float h[8], l[8];
        tmem_ld8(trow + c, h);
        tmem_ld8(trow + NRP + c, l);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[c + i] = h[i] + l[i];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA of the cluster is past its rings
  // rank j receives rows [j rpr, (j + 1) rpr): recv[src rank][row - j rpr][r], rows NRP + 4 floats apart
  constexpr int RS = NRP + 4;
  const int rpr = (OPT_BM + (int)split - 1) / (int)split;
  float* recv = reinterpret_cast<float*>(smem);
  if (warp >= 4 && warp < 8) {
    const int dst = m / rpr, mm = m - dst * rpr;
    const uint32_t base = cluster_addr(recv, (uint32_t)dst) + (uint32_t)(((rank * rpr + mm) * RS) * 4);
#pragma unroll
    for (int r = 0; r < NRP; r += 4) st_cluster_v4(base + (uint32_t)(r * 4), v[r], v[r + 1], v[r + 2], v[r + 3]);
  }
  cluster_sync_all();  // release / acquire: every partial has landed
  pdl_wait();          // y may still be read by the preceding kernel
  if (!aborted()) {
    // thread: one row mm of this rank's slice and 4 activation rows per item
    // (16-byte shared-memory reads, warp-coalesced stores of y)
    const int j0 = (int)rank * rpr;
    int rows = OPT_BM - j0 < rpr ? OPT_BM - j0 : rpr;
    if (d_model - n0 - j0 < rows) rows = d_model - n0 - j0;
    const int groups = (n_rows + 3) >> 2;
    for (int e = threadIdx.x; e < rows * groups; e += OPT_THREADS) {
      const int g = e / rows, mm = e - g * rows;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t src = 0; src < split; ++src) {
        const float4 t = *reinterpret_cast<const float4*>(recv + (src * rpr + mm) * RS + 4 * g);
        acc.x += t.x;
        acc.y += t.y;
        acc.z += t.z;
        acc.w += t.w;
      }
      float* yc = y + (size_t)(4 * g) * d_model + n0 + j0 + mm;
      const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < n_rows) yc[(size_t)i * d_model] = a4[i];
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
}

// cuTensorMapEncodeTiled from the driver (no link-time dependency on it).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // a driver entry point is process-wide; the static is initialised once (thread-safe)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
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

template <int NRP, bool PACKED>
cudaError_t launch_out_proj_tc(int nr, int d_model, int k_dim, const float* x, const void* w, float* y, unsigned* err,
                               cudaStream_t s) {
  constexpr int smem = opt_smem_bytes(NRP);
  static std::atomic<unsigned long long> attr_set{0};  // one set of per-device flags per kernel instance
  const cudaError_t ea = smem_limit_once(attr_set, out_proj_tc_kernel<NRP, PACKED>, smem);
  if (ea != cudaSuccess) return ea;
  CUtensorMap tw;
  memset(&tw, 0, sizeof(tw));
  if (!PACKED && !encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, d_model, k_dim, OPT_BK, OPT_BM))
    return cudaErrorNotSupported;
  // K split (the cluster size): about opt_ctas_per_sm CTAs per SM, at most 8, at most one per K stage
  const int n_mt = (d_model + OPT_BM - 1) / OPT_BM;
  const int n_kb = (k_dim + OPT_BK - 1) / OPT_BK;
  int split = opt_ctas_per_sm(NRP) * device_sm_count() / n_mt;
  if (split > 8) split = 8;
  if (split > n_kb) split = n_kb;
  if (split < 1) split = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_mt, split);
  cfg.blockDim = dim3(OPT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = split;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, out_proj_tc_kernel<NRP, PACKED>, tw,
                                           PACKED ? static_cast<const uint8_t*>(w) : nullptr, x, nr, d_model, k_dim,
                                           y, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool PACKED>
static cudaError_t out_proj_tc_passes(int n_rows, int d_model, int k_dim, const float* x, const void* w, float* y,
                                      unsigned* err, cudaStream_t s) {
  // tensor-core passes of up to 64 activation rows
  for (int r0 = 0; r0 < n_rows; r0 += 64) {
    const int nr = n_rows - r0 < 64 ? n_rows - r0 : 64;
    const float* xr = x + (size_t)r0 * k_dim;
    float* yr = y + (size_t)r0 * d_model;
    cudaError_t e;
    if (nr <= 8) e = launch_out_proj_tc<8, PACKED>(nr, d_model, k_dim, xr, w, yr, err, s);
    else if (nr <= 16) e = launch_out_proj_tc<16, PACKED>(nr, d_model, k_dim, xr, w, yr, err, s);
    else if (nr <= 32) e = launch_out_proj_tc<32, PACKED>(nr, d_model, k_dim, xr, w, yr, err, s);
    else e = launch_out_proj_tc<64, PACKED>(nr, d_model, k_dim, xr, w, yr, err, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// W (bf16 [d_model][k_dim], row-major) -> the packed box order of out_proj_tc_kernel<., true>:
// thread i writes 16-byte chunk i of the packed buffer: box (row tile T, K stage c), row r,
// swizzled chunk position jj <- source chunk j = jj ^ (r % 8) (8 bf16 of row T 128 + r,
// columns 64 c + 8 j ..); zero past d_model or k_dim.
__global__ void pack_wo_kernel(int d_model, int k_dim, int n_kb, const __nv_bfloat16* __restrict__ w,
                               uint4* __restrict__ out, long long n_chunks) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_chunks) return;
  const int jj = (int)(i & 7), r = (int)((i >> 3) & 127);
  const long long box = i >> 10;
  const int c = (int)(box % n_kb), T = (int)(box / n_kb);
  const int j = jj ^ (r & 7);
  const int row = T * OPT_BM + r, col = c * OPT_BK + 8 * j;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (row < d_model && col < k_dim) v = __ldg(reinterpret_cast<const uint4*>(w + (size_t)row * k_dim + col));
  out[i] = v;
}

size_t wo_packed_bytes(int d_model, int k_dim) {
  return (size_t)((d_model + OPT_BM - 1) / OPT_BM) * ((k_dim + OPT_BK - 1) / OPT_BK) * OPT_WBYTES;
}

cudaError_t launch_pack_wo(int d_model, int k_dim, const void* w, void* out, cudaStream_t s) {
  const int n_kb = (k_dim + OPT_BK - 1) / OPT_BK;
  const long long n_chunks = (long long)wo_packed_bytes(d_model, k_dim) / 16;
  if (n_chunks == 0) return cudaSuccess;
  pack_wo_kernel<<<(unsigned)((n_chunks + 255) / 256), 256, 0, s>>>(
      d_model, k_dim, n_kb, static_cast<const __nv_bfloat16*>(w), static_cast<uint4*>(out), n_chunks);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_packed(int n_rows, int d_model, int k_dim, const float* x, const void* w_packed, float* y,
                                   unsigned* err, cudaStream_t s) {
  if (n_rows == 0 || d_model == 0) return cudaSuccess;
  return out_proj_tc_passes<true>(n_rows, d_model, k_dim, x, w_packed, y, err, s);
}

cudaError_t launch_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                            int w_dtype, float* y, unsigned* err, cudaStream_t s) {
  if (n_rows == 0 || d_model == 0) return cudaSuccess;
  if (w_dtype == KVQ_BF16) return out_proj_tc_passes<false>(n_rows, d_model, k_dim, x, w, y, err, s);
  const dim3 grid((d_model + 31) / 32);
  for (int r0 = 0; r0 < n_rows; r0 += 32) {
    const int nr = n_rows - r0 < 32 ? n_rows - r0 : 32;
    const float* xr = x + (size_t)r0 * k_dim;
    float* yr = y + (size_t)r0 * d_model;
    if (nr <= 8) out_proj_mma_kernel<KVQ_F32, 1><<<grid, 256, 0, s>>>(nr, d_model, k_dim, xr, w, yr);
    else if (nr <= 16) out_proj_mma_kernel<KVQ_F32, 2><<<grid, 256, 0, s>>>(nr, d_model, k_dim, xr, w, yr);
    else out_proj_mma_kernel<KVQ_F32, 4><<<grid, 256, 0, s>>>(nr, d_model, k_dim, xr, w, yr);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvq
