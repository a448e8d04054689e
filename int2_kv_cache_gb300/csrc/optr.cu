// OptR calibration of one KV head on the GPU ("Output-Aware Rotation for INT2
// KV-Cache Quantization", §4.2 Eq. 11, §4.3 Eqs. 12-14, §4.4 Eqs. 15-16, §4.5
// Eqs. 17-18, Algorithm 1; §5 implementation details).
//
// Everything here is fp64: the calibration is an offline step whose arithmetic
// is small next to a decode (one head, a few thousand tokens), and its decisions
// (the INT2 codes inside the straight-through forward pass) must equal the fp64
// reference's for the losses and gradients to agree.
//
// One loss + gradient evaluation (keys):
//   S = A - A^T, E = exp(S), R = R^0 E                          (Eq. 11)
//   z = (k - mu) R, z~ = Q_2(z; c) per token (group of 128), STE mask m = [c min z <= z <= c max z]
//   k~ = z~ R^T                                                  (effective keys)
//   per query position t and query head j of the head:
//     p = softmax_{s<=t}(q k_s / sqrt d), p^K = softmax_{s<=t}(q k~_s / sqrt d)     (Eq. 12)
//     e_K = [(p^K - p)^T V] W_O,j^T                                                (Eq. 13)
//     L_K = mean_{t,j} [ KL(p || p^K) + lambda_K ||e_K||^2 / d_model ]           (Eq. 14)
//   backward: dL/da^K_s = p^K_s (g_s - p^K . g) + (p^K_s - p_s), g_s = v_s . (2 lambda_K / d_model) W_O,j^T e_K;
//   dL/dk~_s = sum_{t,j} dL/da^K_{t,j,s} q_{t,j} / (sqrt d n); through k~ = Q(x R) R^T with the
//   straight-through estimator (Eq. 18): dR = G^T z~ + x^T ((G R) * m);
//   dL/dE = R^0^T dR; dL/dS = L_exp(S^T, dL/dE) (the Frechet derivative of exp, the adjoint of
//   L_exp(S, .)); dL/dA = dL/dS - (dL/dS)^T.
// Values (Eqs. 15-16) likewise with e_V = [p^K^T (V~ - V)] W_O,j^T under the fixed weights of the
// selected key rotation, L_V = mean ||e_V||^2 / d_model.
// e enters only through ||W_j c||^2 = c . M_j c and W_j^T e = M_j c, so the d_model-wide
// products are replaced by the 128 x 128 Gram matrix M_j = W_j^T W_j of each query head,
// formed once per call; the other products are fp64 GEMMs over all pairs at once.
//
// The exponential and its Frechet derivative use scaling and squaring with a
// Taylor series: exp(X) = (T(X / 2^s))^(2^s) with ||X / 2^s||_1 <= 1/2 and 18
// terms (truncation below 1e-20 relative), the derivative carried alongside as
// the upper-right block of exp([[X, E], [0, X]]) (each Taylor term and each
// squaring is a block-triangular product).
#include <cmath>
#include <cstdio>

#include "async_copy.cuh"
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr double INV_SQRT_D64 = 0.08838834764831845;  // 1 / sqrt(128)
constexpr int TAYLOR_TERMS = 18;
constexpr int MAX_SQUARINGS = 40;  // ||S||_1 up to 2^39: beyond that the call reports an error

// ---------------------------------------------------------------------------
// fp64 GEMM: C = alpha op(A) op(B) + beta C, row-major, op = transpose or not.
// With `skip` non-null and *skip <= step, the kernel copies `copy_src` into C
// instead (the data-dependent number of squarings of the exponential).
//
// The matrices here are small (128 x 128, or a few thousand rows by 128) and the
// part's fp64 rate is about two FMAs per clock per SM, so the work is spread over
// every SM: 16 x 16 output tiles, one output per thread, and when the tiles are
// fewer than the SMs the K range is split over a cluster of up to 8 blocks.  Each
// block stores its partial tile into the first block's shared memory (distributed
// shared memory), which adds them in rank order: the result does not depend on timing.
// ---------------------------------------------------------------------------
constexpr int GT = 16;            // output tile edge
constexpr int GK = 32;            // k-step staged in shared memory
constexpr int GEMM_MAX_SPLIT = 8;  // blocks of a cluster splitting K

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store v at the address of `local` in the shared memory of cluster block `rank`.
__device__ __forceinline__ void st_cluster_f64(const double* local, unsigned rank, double v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(remote), "d"(v) : "memory");
}

template <typename TA, typename TB>  // operand types (fp64, or fp32 widened on load)
__global__ void __launch_bounds__(GT * GT) gemm_f64_kernel(int M, int N, int K, double alpha,
                                                          const TA* __restrict__ A, int lda, int ta,
                                                          const TB* __restrict__ B, int ldb, int tb, double beta,
                                                          double* __restrict__ C, int ldc, int split,
                                                          const int* __restrict__ skip, int step,
                                                          const double* __restrict__ copy_src) {
  __shared__ double As[GK][GT + 1];  // As[k][m]
  __shared__ double Bs[GK][GT + 1];  // Bs[k][n]
  __shared__ double red[GEMM_MAX_SPLIT][GT * GT];
  const int tid = threadIdx.x, tx = tid % GT, ty = tid / GT;
  const int m0 = blockIdx.y * GT, n0 = blockIdx.x * GT;
  const int m = m0 + ty, n = n0 + tx;
  const unsigned rank = split > 1 ? cluster_rank() : 0u;
  if (skip && *skip <= step) {  // the same decision in every block of the cluster
    if (rank == 0 && m < M && n < N) C[(size_t)m * ldc + n] = copy_src[(size_t)m * ldc + n];
    return;
  }
  // this block's K range
  const int kc = (K + split - 1) / split;
  const int k_lo = min(K, (int)rank * kc), k_hi = min(K, k_lo + kc);
  double acc = 0.0;
  for (int k0 = k_lo; k0 < k_hi; k0 += GK) {
    for (int i = tid; i < GT * GK; i += GT * GT) {
      // element (mm, kk) of the A tile; consecutive threads take consecutive addresses
      const int mm = ta ? i % GT : i / GK, kk = ta ? i / GT : i % GK;
      const int am = m0 + mm, ak = k0 + kk;
      As[kk][mm] = (am < M && ak < k_hi) ? (double)(ta ? A[(size_t)ak * lda + am] : A[(size_t)am * lda + ak]) : 0.0;
      const int nn = tb ? i / GK : i % GT, kb = tb ? i % GK : i / GT;
      const int bn = n0 + nn, bk = k0 + kb;
      Bs[kb][nn] = (bn < N && bk < k_hi) ? (double)(tb ? B[(size_t)bn * ldb + bk] : B[(size_t)bk * ldb + bn]) : 0.0;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < GK; ++kk) acc = fma(As[kk][ty], Bs[kk][tx], acc);
    __syncthreads();
  }
  if (split > 1) {
    cluster_barrier();  // every block of the cluster has started: its shared memory exists
    if (rank == 0) red[0][tid] = acc;
    else st_cluster_f64(&red[rank][tid], 0u, acc);
    cluster_barrier();  // release / acquire: every partial has landed in the first block
    if (rank != 0) return;
    acc = red[0][tid];
    for (int r = 1; r < split; ++r) acc += red[r][tid];
  }
  if (m < M && n < N) {
    double* c = C + (size_t)m * ldc + n;
    *c = beta == 0.0 ? alpha * acc : fma(alpha, acc, beta * *c);
  }
}

template <typename TA, typename TB>
cudaError_t gemm64(cudaStream_t s, int M, int N, int K, double alpha, const TA* A, int lda, bool ta, const TB* B,
                   int ldb, bool tb, double beta, double* C, int ldc, const int* skip = nullptr, int step = 0,
                   const double* copy_src = nullptr) {
  const int tiles = ((N + GT - 1) / GT) * ((M + GT - 1) / GT);
  int split = 1;
  while (tiles * split < device_sm_count() && split < GEMM_MAX_SPLIT && K >= 2 * split * GK) split *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + GT - 1) / GT, (M + GT - 1) / GT, split);
  cfg.blockDim = dim3(GT * GT);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = split;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_f64_kernel<TA, TB>, M, N, K, alpha, A, lda, ta ? 1 : 0, B, ldb, tb ? 1 : 0,
                            beta, C, ldc, split, skip, step, copy_src);
}

// ---------------------------------------------------------------------------
// Small elementwise kernels on 128 x 128 matrices (one CTA of 256 threads or a grid).
// ---------------------------------------------------------------------------
constexpr int NN = D * D;

// S = A - A^T (or its transpose when `transposed`: S^T = A^T - A).
__global__ void skew_kernel(const double* __restrict__ a, double* __restrict__ s, int transposed) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= NN) return;
  const int r = i / D, c = i % D;
  const double v = a[r * D + c] - a[c * D + r];
  s[i] = transposed ? -v : v;
}

// The number of squarings for X (1-norm = max column sum): s = smallest with
// ||X||_1 / 2^s <= 1/2; X_s = X / 2^s and (optionally) E_s = E / 2^s; F = I + X_s,
// L = E_s (the first Taylor term), T = X_s, Dk = E_s.  One CTA of 256 threads.
__global__ void expm_setup_kernel(const double* __restrict__ x, const double* __restrict__ e, double* __restrict__ xs,
                                  double* __restrict__ es, double* __restrict__ f, double* __restrict__ l,
                                  double* __restrict__ t, double* __restrict__ dk, int* __restrict__ n_sq,
                                  unsigned* err) {
  __shared__ double colmax[256];
  __shared__ int s_sq;
  const int tid = threadIdx.x;
  double m = 0.0;
  for (int c = tid; c < D; c += 256) {
    double sum = 0.0;
    for (int r = 0; r < D; ++r) sum += fabs(x[r * D + c]);
    m = fmax(m, sum);
  }
  colmax[tid] = m;
  __syncthreads();
  if (tid == 0) {
    double nrm = 0.0;
    for (int i = 0; i < 256; ++i) nrm = fmax(nrm, colmax[i]);
    int sq = 0;
    while (sq < MAX_SQUARINGS && nrm > 0.5) {
      nrm *= 0.5;
      ++sq;
    }
    if (nrm > 0.5 || !(nrm == nrm)) flag_error(err, ERR_SEQ_RANGE);  // a generator too large (or not finite)
    s_sq = sq;
    *n_sq = sq;
  }
  __syncthreads();
  const double sc = ldexp(1.0, -s_sq);
  for (int i = tid; i < NN; i += 256) {
    const double v = x[i] * sc;
    xs[i] = v;
    t[i] = v;
    f[i] = v + ((i / D) == (i % D) ? 1.0 : 0.0);
    if (e) {
      const double w = e[i] * sc;
      es[i] = w;
      dk[i] = w;
      l[i] = w;
    }
  }
}

__global__ void axpy_kernel(int n, const double* __restrict__ x, double* __restrict__ y) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] += x[i];
}

// out = g - g^T (the gradient with respect to A of a function of S = A - A^T)
__global__ void antisym_kernel(const double* __restrict__ g, double* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= NN) return;
  const int r = i / D, c = i % D;
  out[i] = g[r * D + c] - g[c * D + r];
}

// Adam (common defaults; bias-corrected moments passed as 1 - beta^t)
__global__ void adam_kernel(double* __restrict__ a, const double* __restrict__ g, double* __restrict__ m,
                            double* __restrict__ v, double lr, double b1, double b2, double eps, double c1, double c2) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= NN) return;
  const double gi = g[i];
  const double mi = b1 * m[i] + (1.0 - b1) * gi;
  const double vi = b2 * v[i] + (1.0 - b2) * gi * gi;
  m[i] = mi;
  v[i] = vi;
  const double mh = mi / c1, vh = vi / c2;
  a[i] = a[i] - lr * mh / (sqrt(vh) + eps);
}

// Selection: a strictly lower score replaces the best (ties keep the earlier candidate).
__global__ void select_kernel(const double* __restrict__ score, double* __restrict__ best,
                              const double* __restrict__ a, double* __restrict__ best_a, int first) {
  const bool take = first || *score < *best;
  __syncthreads();
  if (!take) return;
  for (int i = threadIdx.x; i < NN; i += blockDim.x) best_a[i] = a[i];
  if (threadIdx.x == 0) *best = *score;
}

__global__ void fill_kernel(int n, double v, double* __restrict__ y) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = v;
}

// fp32 -> fp64 rows, optionally minus a per-channel mean: y[r][c] = x[r][c] - mu[c]
__global__ void widen_kernel(int n, const float* __restrict__ x, const float* __restrict__ mu, double* __restrict__ y) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  y[i] = (double)x[i] - (mu ? (double)mu[i % D] : 0.0);
}

// ---------------------------------------------------------------------------
// Q_2 in the loop (Eq. 4 forward, Eq. 18 straight-through): one warp per row of
// 128 values z: lo = c min z, hi = c max z, scale = fp16_rn((hi - lo) / 3),
// zero = fp16_rn(lo), code = clamp(rint_even((z - zero) / scale), 0, 3) (0 for a
// zero scale); zq = zero + scale code; mask = 1 where lo <= z <= hi.
// ---------------------------------------------------------------------------
__global__ void quant_ste_kernel(int n_rows, const double* __restrict__ z, double clip, double* __restrict__ zq,
                                 double* __restrict__ mask) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= n_rows) return;
  const double* zr = z + (size_t)warp * D;
  double v[4];
  double mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = zr[4 * lane + i];
    mn = fmin(mn, v[i]);
    mx = fmax(mx, v[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const double lo = clip * mn, hi = clip * mx;
  const double s = (double)__half2float(__double2half((hi - lo) / 3.0));
  const double z0 = (double)__half2float(__double2half(lo));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    double c = 0.0;
    if (s > 0.0) c = fmin(fmax(rint((v[i] - z0) / s), 0.0), 3.0);
    zq[(size_t)warp * D + 4 * lane + i] = z0 + s * c;
    mask[(size_t)warp * D + 4 * lane + i] = (v[i] >= lo && v[i] <= hi) ? 1.0 : 0.0;
  }
}

// dst = src * mask (elementwise)
__global__ void mask_mul_kernel(int n, const double* __restrict__ src, const double* __restrict__ mask,
                                double* __restrict__ dst) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = src[i] * mask[i];
}

// ---------------------------------------------------------------------------
// Row kernels over the (query position, query head) pairs of the head, one CTA of
// 256 threads per pair: pair pr = i * G + j <-> position t = n_tok - n_qpos + i
// (causal: a row's entries s > t are zero).  The products around them are fp64
// GEMMs: logits Q K^T / sqrt(d), C = (P^K - P) V (keys) or P^K (V~ - V) (values),
// U = C_j M_j with the Gram matrix M_j = W_j^T W_j of the head's W_O columns
// (so e = W_j c never has to be formed: ||e||^2 = c . M_j c and W_j^T e = M_j c),
// and G = U V^T.
// ---------------------------------------------------------------------------
__device__ __forceinline__ double block_reduce(double v, double* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmax(v, w) : v + w;
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double r = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = is_max ? fmax(r, red[w]) : r + red[w];
  return r;
}

// log-sum-exp of row[0 .. t] (the whole block gets it)
__device__ __forceinline__ double row_lse(const double* row, int t, double* red) {
  double m = -INFINITY;
  for (int s = threadIdx.x; s <= t; s += blockDim.x) m = fmax(m, row[s]);
  m = block_reduce(m, red, true);
  double sum = 0.0;
  for (int s = threadIdx.x; s <= t; s += blockDim.x) sum += exp(row[s] - m);
  sum = block_reduce(sum, red, false);
  return m + log(sum);
}

// Causal log-softmax of the raw logits in place: log p_s for s <= t (the reference
// softmax of Eq. 12, fixed for a trace).
__global__ void __launch_bounds__(256) log_softmax_rows_kernel(int n_tok, int n_qpos, int gqa, double* __restrict__ a) {
  __shared__ double red[8];
  const int pr = blockIdx.x, t = n_tok - n_qpos + pr / gqa;
  double* row = a + (size_t)pr * n_tok;
  const double lse = row_lse(row, t, red);
  for (int s = threadIdx.x; s <= t; s += blockDim.x) row[s] -= lse;
}

// p^K = softmax of the effective-key logits a (Eq. 12).  With weights_out: p^K into it
// (the value phase's fixed weights).  Otherwise a <- p^K, d <- p^K - p and
// kl[pr] = sum_{s<=t} p_s (log p_s - log p^K_s) (Eq. 14's first term), p = exp(logp).
__global__ void __launch_bounds__(256) key_rows_kernel(int n_tok, int n_qpos, int gqa, double* __restrict__ a,
                                                       const double* __restrict__ logp, double* __restrict__ d,
                                                       double* __restrict__ kl, double* __restrict__ weights_out) {
  __shared__ double red[8];
  const int pr = blockIdx.x, t = n_tok - n_qpos + pr / gqa;
  double* row = a + (size_t)pr * n_tok;
  const double lse = row_lse(row, t, red);
  if (weights_out) {
    for (int s = threadIdx.x; s < n_tok; s += blockDim.x)
      weights_out[(size_t)pr * n_tok + s] = s <= t ? exp(row[s] - lse) : 0.0;
    return;
  }
  const double* lp = logp + (size_t)pr * n_tok;
  double* dr = d + (size_t)pr * n_tok;
  double k = 0.0;
  for (int s = threadIdx.x; s < n_tok; s += blockDim.x) {
    if (s <= t) {
      const double lq = row[s] - lse, pk = exp(lq), p = exp(lp[s]);
      k += p * (lp[s] - lq);
      row[s] = pk;
      dr[s] = pk - p;
    } else {
      row[s] = 0.0;
      dr[s] = 0.0;
    }
  }
  k = block_reduce(k, red, false);
  if (threadIdx.x == 0) kl[pr] = k;
}

// lossp[pr] = (kl[pr] + c_pr . u_pr / 2) * scale (kl absent: 0); one warp per pair.
// With u = (2 lambda / d_model) M_j c, c . u / 2 = lambda ||W_j c||^2 / d_model.
__global__ void pair_loss_kernel(int np, const double* __restrict__ c, const double* __restrict__ u,
                                 const double* __restrict__ kl, double scale, double* __restrict__ lossp) {
  const int pr = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (pr >= np) return;
  double v = 0.0;
#pragma unroll
  for (int i = 0; i < 4; ++i) v = fma(c[(size_t)pr * D + 4 * lane + i], u[(size_t)pr * D + 4 * lane + i], v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) lossp[pr] = ((kl ? kl[pr] : 0.0) + 0.5 * v) * scale;
}

// dL/da^K_s = (p^K_s (g_s - p^K . g) + (p^K_s - p_s)) / n for s <= t, 0 beyond
// (the softmax and KL backward; g = U V^T row).
__global__ void __launch_bounds__(256) key_grad_rows_kernel(int n_tok, int n_qpos, int gqa,
                                                            const double* __restrict__ pk,
                                                            const double* __restrict__ g,
                                                            const double* __restrict__ logp, double inv_n,
                                                            double* __restrict__ da) {
  __shared__ double red[8];
  const int pr = blockIdx.x, t = n_tok - n_qpos + pr / gqa;
  const size_t r0 = (size_t)pr * n_tok;
  double pg = 0.0;
  for (int s = threadIdx.x; s <= t; s += blockDim.x) pg = fma(pk[r0 + s], g[r0 + s], pg);
  pg = block_reduce(pg, red, false);
  for (int s = threadIdx.x; s < n_tok; s += blockDim.x)
    da[r0 + s] = s <= t ? (pk[r0 + s] * (g[r0 + s] - pg) + (pk[r0 + s] - exp(logp[r0 + s]))) * inv_n : 0.0;
}

// loss = sum of the per-pair terms in pair order (deterministic); optionally also into hist[idx]
__global__ void sum_loss_kernel(int np, const double* __restrict__ lp, double* __restrict__ loss,
                                double* __restrict__ hist, int idx) {
  if (threadIdx.x != 0) return;
  double s = 0.0;
  for (int i = 0; i < np; ++i) s += lp[i];
  if (loss) *loss = s;
  if (hist) hist[idx] = s;
}

// dst = a - b (elementwise)
__global__ void sub_kernel(int n, const double* __restrict__ a, const double* __restrict__ b, double* __restrict__ dst) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = a[i] - b[i];
}

// ---------------------------------------------------------------------------
// Workspace: 128 x 128 matrices, per-token temporaries, the widened inputs of the
// training trace and of the held-out trace, per-pair buffers, scalars.
// ---------------------------------------------------------------------------
struct OptrTrace {  // one trace, widened to fp64
  int n_tok, n_qpos;
  double *x, *kraw, *vv, *q, *pair;  // x = k - mu; pair: [pairs][n_tok] (dL/da^K, or the fixed weights p^K)
  double* logp;                      // [pairs][n_tok]: log p of the raw keys (fixed for the trace)
};

struct OptrWs {
  double *S, *E, *R, *xs, *es, *F, *L, *T, *Dk, *T2, *D2, *F2, *L2, *dR, *dE, *G, *m, *v, *a, *best_a, *outF, *gA;
  double *z, *zq, *mask, *keff, *geff, *dzq;  // [n_tok][128], n_tok the larger trace's
  double *u, *lossp;                         // [pairs][128], [pairs]
  double *ak, *dm, *cm, *kl;                 // [pairs][n_tok] x 2, [pairs][128], [pairs]
  double* gram;                              // [gqa][128][128]: M_j = W_j^T W_j
  double* scal;                              // [0] loss, [1] score, [2] best score
  int* nsq;
  OptrTrace tr, ho;                          // training and held-out traces
};

size_t optr_ws_layout(void* base, int n_tok, int n_qpos, int n_tok_h, int n_qpos_h, int gqa, OptrWs* o) {
  const size_t np = (size_t)n_qpos * gqa, nph = (size_t)n_qpos_h * gqa;
  const size_t ntm = (size_t)(n_tok > n_tok_h ? n_tok : n_tok_h), npm = np > nph ? np : nph;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = (off + bytes + 255) & ~size_t(255);
    return at;
  };
  size_t mats[22], toks[6], tr[6], ho[6];
  for (int i = 0; i < 22; ++i) mats[i] = take(NN * sizeof(double));
  for (int i = 0; i < 6; ++i) toks[i] = take(ntm * D * sizeof(double));
  const size_t o_u = take(npm * D * sizeof(double));
  const size_t o_lp = take(npm * sizeof(double));
  const size_t o_ak = take(npm * ntm * sizeof(double));
  const size_t o_dm = take(npm * ntm * sizeof(double));
  const size_t o_cm = take(npm * D * sizeof(double));
  const size_t o_kl = take(npm * sizeof(double));
  const size_t o_gram = take((size_t)gqa * NN * sizeof(double));
  const size_t o_sc = take(4 * sizeof(double));
  const size_t o_nsq = take(4 * sizeof(int));
  for (int i = 0; i < 3; ++i) tr[i] = take((size_t)n_tok * D * sizeof(double));
  tr[3] = take(np * D * sizeof(double));
  tr[4] = take(np * n_tok * sizeof(double));
  tr[5] = take(np * n_tok * sizeof(double));
  for (int i = 0; i < 3; ++i) ho[i] = take((size_t)n_tok_h * D * sizeof(double));
  ho[3] = take(nph * D * sizeof(double));
  ho[4] = take(nph * n_tok_h * sizeof(double));
  ho[5] = take(nph * n_tok_h * sizeof(double));
  if (o) {
    char* p = static_cast<char*>(base);
    double** mp[22] = {&o->S, &o->E, &o->R, &o->xs, &o->es, &o->F, &o->L, &o->T, &o->Dk, &o->T2, &o->D2,
                       &o->F2, &o->L2, &o->dR, &o->dE, &o->G, &o->m, &o->v, &o->a, &o->best_a, &o->outF, &o->gA};
    for (int i = 0; i < 22; ++i) *mp[i] = reinterpret_cast<double*>(p + mats[i]);
    double** tp[6] = {&o->z, &o->zq, &o->mask, &o->keff, &o->geff, &o->dzq};
    for (int i = 0; i < 6; ++i) *tp[i] = reinterpret_cast<double*>(p + toks[i]);
    o->u = reinterpret_cast<double*>(p + o_u);
    o->lossp = reinterpret_cast<double*>(p + o_lp);
    o->ak = reinterpret_cast<double*>(p + o_ak);
    o->dm = reinterpret_cast<double*>(p + o_dm);
    o->cm = reinterpret_cast<double*>(p + o_cm);
    o->kl = reinterpret_cast<double*>(p + o_kl);
    o->gram = reinterpret_cast<double*>(p + o_gram);
    o->scal = reinterpret_cast<double*>(p + o_sc);
    o->nsq = reinterpret_cast<int*>(p + o_nsq);
    OptrTrace* t2[2] = {&o->tr, &o->ho};
    const size_t* offs[2] = {tr, ho};
    for (int k = 0; k < 2; ++k) {
      t2[k]->n_tok = k ? n_tok_h : n_tok;
      t2[k]->n_qpos = k ? n_qpos_h : n_qpos;
      t2[k]->x = reinterpret_cast<double*>(p + offs[k][0]);
      t2[k]->kraw = reinterpret_cast<double*>(p + offs[k][1]);
      t2[k]->vv = reinterpret_cast<double*>(p + offs[k][2]);
      t2[k]->q = reinterpret_cast<double*>(p + offs[k][3]);
      t2[k]->pair = reinterpret_cast<double*>(p + offs[k][4]);
      t2[k]->logp = reinterpret_cast<double*>(p + offs[k][5]);
    }
  }
  return off;
}

#define KVQ_TRY(x)                        \
  do {                                    \
    const cudaError_t e_ = (x);           \
    if (e_ != cudaSuccess) return e_;     \
  } while (0)

inline int blocks(size_t n, int t = 256) { return (int)((n + t - 1) / t); }

// exp(X) into outF, and with E non-null also outL = L_exp(X, E).  X, E are 128 x 128
// and must not be workspace matrices that this routine uses (xs .. L2).
cudaError_t expm_pair(const OptrWs& w, const double* X, const double* E, double* outF, double* outL, unsigned* err,
                      cudaStream_t s) {
  expm_setup_kernel<<<1, 256, 0, s>>>(X, E, w.xs, w.es, w.F, w.L, w.T, w.Dk, w.nsq, err);
  KVQ_TRY(cudaGetLastError());
  double *T = w.T, *Dk = w.Dk, *T2 = w.T2, *D2 = w.D2;
  for (int kk = 2; kk <= TAYLOR_TERMS; ++kk) {
    const double inv = 1.0 / kk;
    // D_k = (D_{k-1} X + T_{k-1} E) / k, then T_k = T_{k-1} X / k
    if (E) {
      KVQ_TRY(gemm64(s, D, D, D, inv, Dk, D, false, w.xs, D, false, 0.0, D2, D));
      KVQ_TRY(gemm64(s, D, D, D, inv, T, D, false, w.es, D, false, 1.0, D2, D));
    }
    KVQ_TRY(gemm64(s, D, D, D, inv, T, D, false, w.xs, D, false, 0.0, T2, D));
    axpy_kernel<<<blocks(NN), 256, 0, s>>>(NN, T2, w.F);
    if (E) axpy_kernel<<<blocks(NN), 256, 0, s>>>(NN, D2, w.L);
    KVQ_TRY(cudaGetLastError());
    double* tmp = T; T = T2; T2 = tmp;
    tmp = Dk; Dk = D2; D2 = tmp;
  }
  // squarings: (F, L) <- (F F, F L + L F), as many as the setup chose (the others copy)
  double *F = w.F, *L = w.L, *F2 = w.F2, *L2 = w.L2;
  for (int st = 0; st < MAX_SQUARINGS; ++st) {
    if (E) {
      KVQ_TRY(gemm64(s, D, D, D, 1.0, F, D, false, L, D, false, 0.0, L2, D, w.nsq, st, L));
      KVQ_TRY(gemm64(s, D, D, D, 1.0, L, D, false, F, D, false, 1.0, L2, D, w.nsq, st, L2));
    }
    KVQ_TRY(gemm64(s, D, D, D, 1.0, F, D, false, F, D, false, 0.0, F2, D, w.nsq, st, F));
    double* tmp = F; F = F2; F2 = tmp;
    tmp = L; L = L2; L2 = tmp;
  }
  KVQ_TRY(cudaMemcpyAsync(outF, F, NN * sizeof(double), cudaMemcpyDeviceToDevice, s));
  if (E && outL) KVQ_TRY(cudaMemcpyAsync(outL, L, NN * sizeof(double), cudaMemcpyDeviceToDevice, s));
  return cudaSuccess;
}

// R = R0 exp(A - A^T) into w.R (w.S holds S)
cudaError_t rotation_of(const OptrWs& w, const double* r0, const double* a, unsigned* err, cudaStream_t s) {
  skew_kernel<<<blocks(NN), 256, 0, s>>>(a, w.S, 0);
  KVQ_TRY(cudaGetLastError());
  KVQ_TRY(expm_pair(w, w.S, nullptr, w.E, nullptr, err, s));
  return gemm64(s, D, D, D, 1.0, r0, D, false, w.E, D, false, 0.0, w.R, D);
}

// Effective rows Q_2(X R) R^T into w.keff (z, zq, mask kept for the backward pass); w.R set.
cudaError_t effective_rows(const OptrWs& w, const double* X, int n_tok, double clip, cudaStream_t s) {
  KVQ_TRY(gemm64(s, n_tok, D, D, 1.0, X, D, false, w.R, D, false, 0.0, w.z, D));
  quant_ste_kernel<<<blocks((size_t)n_tok * 32), 256, 0, s>>>(n_tok, w.z, clip, w.zq, w.mask);
  KVQ_TRY(cudaGetLastError());
  return gemm64(s, n_tok, D, D, 1.0, w.zq, D, false, w.R, D, true, 0.0, w.keff, D);
}

}  // namespace

// ---------------------------------------------------------------------------
// Entry points (kvq_internal.cuh)
// ---------------------------------------------------------------------------
size_t optr_workspace_bytes(int n_tok, int n_qpos, int n_tok_h, int n_qpos_h, int gqa) {
  return optr_ws_layout(nullptr, n_tok, n_qpos, n_tok_h, n_qpos_h, gqa, nullptr);
}

namespace {

cudaError_t widen_trace(const OptrTrace& t, int gqa, const float* q, const float* k, const float* v, const float* mu,
                        cudaStream_t s) {
  const size_t nt = (size_t)t.n_tok * D, nq = (size_t)t.n_qpos * gqa * D;
  widen_kernel<<<blocks(nt), 256, 0, s>>>((int)nt, k, mu, t.x);
  widen_kernel<<<blocks(nt), 256, 0, s>>>((int)nt, k, nullptr, t.kraw);
  widen_kernel<<<blocks(nt), 256, 0, s>>>((int)nt, v, nullptr, t.vv);
  widen_kernel<<<blocks(nq), 256, 0, s>>>((int)nq, q, nullptr, t.q);
  return cudaGetLastError();
}

// log p of the raw keys for every pair of trace t (Eq. 12's reference softmax, fixed for the trace)
cudaError_t raw_logp(const OptrTrace& t, int gqa, cudaStream_t s) {
  const int np = t.n_qpos * gqa;
  KVQ_TRY(gemm64(s, np, t.n_tok, D, INV_SQRT_D64, t.q, D, false, t.kraw, D, true, 0.0, t.logp, t.n_tok));
  log_softmax_rows_kernel<<<np, 256, 0, s>>>(t.n_tok, t.n_qpos, gqa, t.logp);
  return cudaGetLastError();
}

// M_j = W_j^T W_j for the head's query heads (W_j: the 128 columns of W_O of query head j)
cudaError_t gram_of(const OptrWs& w, int gqa, int d_model, const float* w_o, cudaStream_t s) {
  for (int j = 0; j < gqa; ++j)
    KVQ_TRY(gemm64(s, D, D, d_model, 1.0, w_o + (size_t)j * D, gqa * D, true, w_o + (size_t)j * D, gqa * D, false, 0.0,
                   w.gram + (size_t)j * NN, D));
  return cudaSuccess;
}

// U_j = alpha C_j M_j for every query head j (rows i * G + j of C and U)
cudaError_t gram_apply(const OptrWs& w, int n_qpos, int gqa, double alpha, cudaStream_t s) {
  for (int j = 0; j < gqa; ++j)
    KVQ_TRY(gemm64(s, n_qpos, D, D, alpha, w.cm + (size_t)j * D, gqa * D, false, w.gram + (size_t)j * NN, D, false, 0.0,
                   w.u + (size_t)j * D, gqa * D));
  return cudaSuccess;
}

// p^K of the rotation in w.R for trace t into t.pair (the value phase's fixed weights)
cudaError_t key_weights(const OptrWs& w, const OptrTrace& t, int gqa, double clip, cudaStream_t s) {
  KVQ_TRY(effective_rows(w, t.x, t.n_tok, clip, s));
  const int np = t.n_qpos * gqa;
  KVQ_TRY(gemm64(s, np, t.n_tok, D, INV_SQRT_D64, t.q, D, false, w.keff, D, true, 0.0, w.ak, t.n_tok));
  key_rows_kernel<<<np, 256, 0, s>>>(t.n_tok, t.n_qpos, gqa, w.ak, nullptr, nullptr, nullptr, t.pair);
  return cudaGetLastError();
}

// One loss (+ gradient) evaluation of phase 0 (keys) or 1 (values) at generator a with base r0.
// The loss goes to *loss and, with hist, to hist[idx]; the gradient (dL/dA) to grad when non-null.
// Needs w.gram (gram_of) and, for keys, t.logp (raw_logp).
cudaError_t optr_eval(const OptrWs& w, const OptrTrace& t, int gqa, int d_model, int phase, const double* r0,
                      const double* a, double clip, double lam, double* loss, double* hist, int idx, double* grad,
                      unsigned* err, cudaStream_t s) {
  const int n_tok = t.n_tok, np = t.n_qpos * gqa;
  const double* X = phase ? t.vv : t.x;
  KVQ_TRY(rotation_of(w, r0, a, err, s));
  KVQ_TRY(effective_rows(w, X, n_tok, clip, s));
  if (phase == 0) {
    // p^K from the effective keys, C = (p^K - p) V, U = (2 lambda / d_model) C_j M_j
    KVQ_TRY(gemm64(s, np, n_tok, D, INV_SQRT_D64, t.q, D, false, w.keff, D, true, 0.0, w.ak, n_tok));
    key_rows_kernel<<<np, 256, 0, s>>>(n_tok, t.n_qpos, gqa, w.ak, t.logp, w.dm, w.kl, nullptr);
    KVQ_TRY(cudaGetLastError());
    KVQ_TRY(gemm64(s, np, D, n_tok, 1.0, w.dm, n_tok, false, t.vv, D, false, 0.0, w.cm, D));
    KVQ_TRY(gram_apply(w, t.n_qpos, gqa, 2.0 * lam / d_model, s));
    pair_loss_kernel<<<blocks((size_t)np * 32), 256, 0, s>>>(np, w.cm, w.u, w.kl, 1.0 / np, w.lossp);
  } else {
    // C = p^K (V~ - V), U = (2 / (d_model n)) C_j M_j
    sub_kernel<<<blocks((size_t)n_tok * D), 256, 0, s>>>(n_tok * D, w.keff, t.vv, w.dzq);
    KVQ_TRY(cudaGetLastError());
    KVQ_TRY(gemm64(s, np, D, n_tok, 1.0, t.pair, n_tok, false, w.dzq, D, false, 0.0, w.cm, D));
    KVQ_TRY(gram_apply(w, t.n_qpos, gqa, 2.0 / ((double)d_model * np), s));
    pair_loss_kernel<<<blocks((size_t)np * 32), 256, 0, s>>>(np, w.cm, w.u, nullptr, 1.0, w.lossp);
  }
  KVQ_TRY(cudaGetLastError());
  sum_loss_kernel<<<1, 32, 0, s>>>(np, w.lossp, loss, hist, idx);
  KVQ_TRY(cudaGetLastError());
  if (!grad) return cudaSuccess;
  // dL/dk~ (keys: DA^T Q / sqrt d with DA from G = U V^T, the 1/n in DA) or dL/dv~ (values: P^T U)
  if (phase == 0) {
    KVQ_TRY(gemm64(s, np, n_tok, D, 1.0, w.u, D, false, t.vv, D, true, 0.0, w.dm, n_tok));
    key_grad_rows_kernel<<<np, 256, 0, s>>>(n_tok, t.n_qpos, gqa, w.ak, w.dm, t.logp, 1.0 / np, t.pair);
    KVQ_TRY(cudaGetLastError());
    KVQ_TRY(gemm64(s, n_tok, D, np, INV_SQRT_D64, t.pair, n_tok, true, t.q, D, false, 0.0, w.geff, D));
  } else {
    KVQ_TRY(gemm64(s, n_tok, D, np, 1.0, t.pair, n_tok, true, w.u, D, false, 0.0, w.geff, D));
  }
  // through k~ = Q(X R) R^T with the straight-through mask: dR = G^T z~ + X^T ((G R) * m)
  KVQ_TRY(gemm64(s, D, D, n_tok, 1.0, w.geff, D, true, w.zq, D, false, 0.0, w.dR, D));
  KVQ_TRY(gemm64(s, n_tok, D, D, 1.0, w.geff, D, false, w.R, D, false, 0.0, w.dzq, D));
  mask_mul_kernel<<<blocks((size_t)n_tok * D), 256, 0, s>>>(n_tok * D, w.dzq, w.mask, w.dzq);
  KVQ_TRY(cudaGetLastError());
  KVQ_TRY(gemm64(s, D, D, n_tok, 1.0, X, D, true, w.dzq, D, false, 1.0, w.dR, D));
  // dL/dE = R0^T dR; dL/dS = L_exp(S^T, dL/dE); dL/dA = dL/dS - (dL/dS)^T
  KVQ_TRY(gemm64(s, D, D, D, 1.0, r0, D, true, w.dR, D, false, 0.0, w.dE, D));
  skew_kernel<<<blocks(NN), 256, 0, s>>>(a, w.S, 1);
  KVQ_TRY(cudaGetLastError());
  KVQ_TRY(expm_pair(w, w.S, w.dE, w.outF, w.G, err, s));
  antisym_kernel<<<blocks(NN), 256, 0, s>>>(w.G, grad);
  return cudaGetLastError();
}

// Adam on A from 0 for `steps` steps, candidates every `every` steps (and step 0), scored on the
// held-out trace (the training one when absent); the best generator ends in w.best_a.
cudaError_t optr_phase(const OptrWs& w, bool heldout, int gqa, int d_model, int phase, const double* r0,
                       double clip, double lam, int steps, double lr, int every, double* hist, unsigned* err,
                       cudaStream_t s) {
  const OptrTrace& sc = heldout ? w.ho : w.tr;
  fill_kernel<<<blocks(NN), 256, 0, s>>>(NN, 0.0, w.a);
  fill_kernel<<<blocks(NN), 256, 0, s>>>(NN, 0.0, w.m);
  fill_kernel<<<blocks(NN), 256, 0, s>>>(NN, 0.0, w.v);
  KVQ_TRY(cudaGetLastError());
  KVQ_TRY(optr_eval(w, sc, gqa, d_model, phase, r0, w.a, clip, lam, w.scal + 1, nullptr, 0, nullptr, err, s));
  select_kernel<<<1, 256, 0, s>>>(w.scal + 1, w.scal + 2, w.a, w.best_a, 1);
  KVQ_TRY(cudaGetLastError());
  const double b1 = 0.9, b2 = 0.999, eps = 1e-8;
  double p1 = 1.0, p2 = 1.0;
  for (int i = 1; i <= steps; ++i) {
    KVQ_TRY(optr_eval(w, w.tr, gqa, d_model, phase, r0, w.a, clip, lam, w.scal, hist, i - 1, w.gA, err, s));
    p1 *= b1;
    p2 *= b2;
    adam_kernel<<<blocks(NN), 256, 0, s>>>(w.a, w.gA, w.m, w.v, lr, b1, b2, eps, 1.0 - p1, 1.0 - p2);
    KVQ_TRY(cudaGetLastError());
    if (every > 0 && i % every == 0) {
      KVQ_TRY(optr_eval(w, sc, gqa, d_model, phase, r0, w.a, clip, lam, w.scal + 1, nullptr, 0, nullptr, err, s));
      select_kernel<<<1, 256, 0, s>>>(w.scal + 1, w.scal + 2, w.a, w.best_a, 0);
      KVQ_TRY(cudaGetLastError());
    }
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_optr_loss_grad(int phase, const OptrTraceIn& tr, int gqa, int d_model, const float* w_o,
                                  const float* mu, const double* r0, const double* a, const double* r_k_sel,
                                  float clip_k, float clip_v, float lam, double* loss, double* grad, void* ws,
                                  unsigned* err, cudaStream_t s) {
  OptrWs w;
  optr_ws_layout(ws, tr.n_tok, tr.n_qpos, 0, 0, gqa, &w);
  KVQ_TRY(widen_trace(w.tr, gqa, tr.q, tr.k, tr.v, mu, s));
  KVQ_TRY(gram_of(w, gqa, d_model, w_o, s));
  if (phase == 0) KVQ_TRY(raw_logp(w.tr, gqa, s));
  if (phase == 1) {  // the fixed weights p^K of the selected key rotation
    KVQ_TRY(cudaMemcpyAsync(w.R, r_k_sel, NN * sizeof(double), cudaMemcpyDeviceToDevice, s));
    KVQ_TRY(key_weights(w, w.tr, gqa, clip_k, s));
  }
  return optr_eval(w, w.tr, gqa, d_model, phase, r0, a, phase ? clip_v : clip_k, lam, loss, nullptr, 0, grad, err,
                   s);
}

cudaError_t launch_optr_calibrate(const OptrTraceIn& tr, const OptrTraceIn* ho, int gqa, int d_model,
                                  const float* w_o, const float* mu, const double* r_k0, const double* r_v0,
                                  float clip_k, float clip_v, float lam, int steps, float lr, int every, double* r_k,
                                  double* r_v, double* loss_k, double* loss_v, void* ws, unsigned* err,
                                  cudaStream_t s) {
  OptrWs w;
  optr_ws_layout(ws, tr.n_tok, tr.n_qpos, ho ? ho->n_tok : 0, ho ? ho->n_qpos : 0, gqa, &w);
  KVQ_TRY(widen_trace(w.tr, gqa, tr.q, tr.k, tr.v, mu, s));
  if (ho) KVQ_TRY(widen_trace(w.ho, gqa, ho->q, ho->k, ho->v, mu, s));
  KVQ_TRY(gram_of(w, gqa, d_model, w_o, s));
  KVQ_TRY(raw_logp(w.tr, gqa, s));
  if (ho) KVQ_TRY(raw_logp(w.ho, gqa, s));
  // keys (Algorithm 1, first loop), then the selected rotation R_K and its weights p^K
  KVQ_TRY(optr_phase(w, ho != nullptr, gqa, d_model, 0, r_k0, clip_k, lam, steps, lr, every, loss_k, err, s));
  KVQ_TRY(rotation_of(w, r_k0, w.best_a, err, s));
  KVQ_TRY(cudaMemcpyAsync(r_k, w.R, NN * sizeof(double), cudaMemcpyDeviceToDevice, s));
  KVQ_TRY(key_weights(w, w.tr, gqa, clip_k, s));
  if (ho) KVQ_TRY(key_weights(w, w.ho, gqa, clip_k, s));
  // values under the selected key path (second loop)
  KVQ_TRY(optr_phase(w, ho != nullptr, gqa, d_model, 1, r_v0, clip_v, 0.0, steps, lr, every, loss_v, err, s));
  KVQ_TRY(rotation_of(w, r_v0, w.best_a, err, s));
  return cudaMemcpyAsync(r_v, w.R, NN * sizeof(double), cudaMemcpyDeviceToDevice, s);
}

}  // namespace kvq
