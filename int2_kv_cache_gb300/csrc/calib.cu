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
#include <algorithm>

#include "quant_common.cuh"

namespace kvq {



struct CalibWs {
  float *qf, *qr, *kf, *vf, *xk_hi, *xk_lo, *xv_hi, *xv_lo, *kq, *vq, *o_rot, *o_ref, *o_un, *gram, *part;
  double* gpart;  // [n_groups][(gd / 32)^2] quadratic-form partials
  double* qsum;   // [5][H_q] per-query-head sums of the error report
  // the sweep's quantized trace as a page pool read by the decode kernels: one
  // "sequence" per calibration position i (the causal prefix of n_tok - n_qpos + i + 1
  // tokens), every sequence's block-table row pointing at the same pages
  uint8_t* pool;
  int32_t *table, *lens;
  void* dws;  // decode workspace
  int n_ctas;
};

constexpr int CA_SPLIT_MAX = 8;  // key splits of the calibration attention

static size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

// Scored groups: n_groups column blocks of gd channels of the attention output
// (joint: one of H_q 128; per KV head: H_kv of G 128; per query head: H_q of 128).
static CalibWs carve(void* ws, int n_tok, int n_qpos, int n_kv_heads, int gqa, int n_groups, int gd,
                     size_t* total) {
  const size_t hq = (size_t)n_kv_heads * gqa;
  const size_t qn = (size_t)n_qpos * hq * D, kn = (size_t)n_tok * n_kv_heads * D;
  const size_t gn = (size_t)n_groups * gd * gd;
  const size_t pn = (size_t)CA_SPLIT_MAX * n_qpos * hq * (D + 4);  // attention partials
  const size_t gpn = 2 * (size_t)n_groups * (gd / 32) * (gd / 32);  // doubles, as float pairs
  const int n_blk = (n_tok + CALIB_PAGE - 1) / CALIB_PAGE;
  const int n_ctas = decode_auto_ctas(n_qpos, n_kv_heads, gqa, n_tok);
  // the pool, block table, lengths and decode workspace, in bytes / 4
  const size_t pooln = (size_t)n_blk * n_kv_heads * 72 * CALIB_PAGE / 4, tabn = (size_t)n_qpos * n_blk;
  const size_t dwn = (decode_workspace_bytes(n_qpos, n_kv_heads, gqa, n_ctas) + 3) / 4;
  const size_t sizes[21] = {qn, qn, kn, kn, kn, kn, kn, kn, kn, kn, qn, qn, qn, gn, pn, gpn, 2 * 5 * hq,
                            pooln, tabn, (size_t)n_qpos, dwn};
  char* p = static_cast<char*>(ws);
  float* ptrs[21];
  size_t off = 0;
  for (int i = 0; i < 21; ++i) {
    ptrs[i] = reinterpret_cast<float*>(p + off);
    off += align_up(sizes[i] * sizeof(float));
  }
  if (total) *total = off;
  return CalibWs{ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[4], ptrs[5], ptrs[6], ptrs[7],
                 ptrs[8], ptrs[9], ptrs[10], ptrs[11], ptrs[12], ptrs[13], ptrs[14],
                 reinterpret_cast<double*>(ptrs[15]), reinterpret_cast<double*>(ptrs[16]),
                 reinterpret_cast<uint8_t*>(ptrs[17]), reinterpret_cast<int32_t*>(ptrs[18]),
                 reinterpret_cast<int32_t*>(ptrs[19]), ptrs[20], n_ctas};
}

// Block table (every row 0 .. n_blk - 1) and prefix lengths of the sweep's decode.
__global__ void calib_pages_kernel(int n_qpos, int n_tok, int n_blk, int32_t* __restrict__ table,
                                   int32_t* __restrict__ lens) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_qpos * n_blk) table[i] = i % n_blk;
  if (i < n_qpos) lens[i] = n_tok - n_qpos + i + 1;
}

static int calib_groups(int n_kv_heads, int joint) { return joint ? 1 : n_kv_heads; }
static int calib_gd(int n_kv_heads, int gqa, int joint) { return (joint ? n_kv_heads * gqa : gqa) * D; }

size_t calib_workspace_bytes(int n_tok, int n_qpos, int n_kv_heads, int gqa, int joint) {
  size_t total = 0;
  carve(nullptr, n_tok, n_qpos, n_kv_heads, gqa, calib_groups(n_kv_heads, joint), calib_gd(n_kv_heads, gqa, joint),
        &total);
  return total;
}

size_t report_workspace_bytes(int n_tok, int n_qpos, int n_kv_heads, int gqa) {
  size_t total = 0;
  carve(nullptr, n_tok, n_qpos, n_kv_heads, gqa, n_kv_heads * gqa, D, &total);
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

// Causal attention, tiled: a CTA takes the G query heads of KV head h at 64 / G
// query positions (64 rows) and a range of keys (one of `split` ranges), and
// streams the keys and values through shared memory 64 tokens at a time
// (cp.async, double-buffered), with an online softmax per row in fp32.
// S = Q K^T: thread (ty, tx) owns rows 4ty..4ty+3 x tokens 4tx..4tx+3; O += P V:
// rows 4ty..4ty+3 x channels 8tx..8tx+7.  With split > 1 each CTA writes the
// row partials (m, l, unnormalised acc) for calib_attn_combine_kernel.
// grid = (n_kv_heads, ceil(n_qpos / (64 / G)), split), block = 256.
constexpr int CA_ROWS = 64, CA_KT = 64, CA_KS = D + 4;  // K rows padded: conflict-free column reads
constexpr int CA_SMEM = (CA_ROWS * D + 2 * CA_KT * CA_KS + 2 * CA_KT * D + CA_ROWS * (CA_KT + 4) + 3 * CA_ROWS) * 4;

__device__ __forceinline__ void ca_cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

template <int G>
__global__ void __launch_bounds__(256, 1) calib_attn_tiled_kernel(int n_tok, int n_qpos, int n_kv_heads, int split,
                                                                  const float* __restrict__ q,
                                                                  const float* __restrict__ k,
                                                                  const float* __restrict__ v, float* __restrict__ o,
                                                                  float* __restrict__ part) {
  constexpr int QB = CA_ROWS / G;  // query positions per CTA
  extern __shared__ __align__(16) float ca_smem[];
  float* sq = ca_smem;                          // [64][128] queries / sqrt(128)
  float* sk = sq + CA_ROWS * D;                 // [2][64][132]
  float* sv = sk + 2 * CA_KT * CA_KS;           // [2][64][128]
  float* sp = sv + 2 * CA_KT * D;               // [64][68] probabilities
  float* sm = sp + CA_ROWS * (CA_KT + 4);       // [64] running max
  float* sl = sm + CA_ROWS;                     // [64] running sum
  float* ss = sl + CA_ROWS;                     // [64] rescale of this tile
  const int h = blockIdx.x, qb0 = blockIdx.y * QB, sidx = blockIdx.z;
  const int hq = n_kv_heads * G;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  // rows r = G * (position - qb0) + head offset
  for (int i = tid; i < CA_ROWS * D / 4; i += 256) {
    const int r = i / (D / 4), c4 = i % (D / 4);
    const int qi = qb0 + r / G, j = h * G + r % G;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (qi < n_qpos) x = reinterpret_cast<const float4*>(q + ((size_t)qi * hq + j) * D)[c4];
    x.x *= INV_SQRT_D; x.y *= INV_SQRT_D; x.z *= INV_SQRT_D; x.w *= INV_SQRT_D;
    reinterpret_cast<float4*>(sq + r * D)[c4] = x;
  }
  if (tid < CA_ROWS) {
    sm[tid] = -INFINITY;
    sl[tid] = 0.f;
  }
  // the keys of this split, limited by the last (causal) position of the CTA's rows
  const int last_q = min(n_qpos, qb0 + QB) - 1;
  const int t_max = n_tok - n_qpos + last_q;  // inclusive
  const int n_tiles_all = (n_tok + CA_KT - 1) / CA_KT;
  const int per = (n_tiles_all + split - 1) / split;
  const int tile0 = sidx * per;
  const int tile1 = min(min(n_tiles_all, tile0 + per), t_max / CA_KT + 1);
  auto load_tile = [&](int tile, int buf) {
    const int s0 = tile * CA_KT;
    for (int i = tid; i < CA_KT * D / 4; i += 256) {
      const int r = i / (D / 4), c4 = i % (D / 4);
      const int s = min(s0 + r, n_tok - 1);  // rows past the end are masked below
      ca_cp16(sk + (buf * CA_KT + r) * CA_KS + 4 * c4, k + ((size_t)s * n_kv_heads + h) * D + 4 * c4);
      ca_cp16(sv + (buf * CA_KT + r) * D + 4 * c4, v + ((size_t)s * n_kv_heads + h) * D + 4 * c4);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[4][8];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
  if (tile0 < tile1) load_tile(tile0, 0);
  __syncthreads();
  for (int tile = tile0; tile < tile1; ++tile) {
    const int buf = (tile - tile0) & 1;
    if (tile + 1 < tile1) {
      load_tile(tile + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    // ---- scores ----
    const float* kb = sk + buf * CA_KT * CA_KS;
    float sc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) sc[a][b] = 0.f;
#pragma unroll 4
    for (int c4 = 0; c4 < D / 4; ++c4) {
      float4 qa[4], kk[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) qa[a] = reinterpret_cast<const float4*>(sq + (4 * ty + a) * D)[c4];
#pragma unroll
      for (int b = 0; b < 4; ++b) kk[b] = reinterpret_cast<const float4*>(kb + (4 * tx + b) * CA_KS)[c4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          sc[a][b] = fmaf(qa[a].x, kk[b].x, sc[a][b]);
          sc[a][b] = fmaf(qa[a].y, kk[b].y, sc[a][b]);
          sc[a][b] = fmaf(qa[a].z, kk[b].z, sc[a][b]);
          sc[a][b] = fmaf(qa[a].w, kk[b].w, sc[a][b]);
        }
    }
    // ---- causal mask, online softmax (16 threads per row group) ----
    const int s0 = tile * CA_KT;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      const int qi = qb0 + r / G;
      const int tpos = n_tok - n_qpos + qi;  // keys s <= tpos
      float mx = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = s0 + 4 * tx + b;
        if (s > tpos || s >= n_tok || qi >= n_qpos) sc[a][b] = -INFINITY;
        mx = fmaxf(mx, sc[a][b]);
      }
#pragma unroll
      for (int m = 1; m < 16; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      const float mold = sm[r];
      const float mnew = fmaxf(mold, mx);
      float psum = 0.f;
      float4 pv;
      float pr[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        pr[b] = mnew == -INFINITY ? 0.f : __expf(sc[a][b] - mnew);
        psum += pr[b];
      }
      pv = make_float4(pr[0], pr[1], pr[2], pr[3]);
      reinterpret_cast<float4*>(sp + r * (CA_KT + 4))[tx] = pv;
#pragma unroll
      for (int m = 1; m < 16; m <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, m);
      __syncwarp();
      if (tx == 0) {
        const float scale = mold == -INFINITY ? 0.f : __expf(mold - mnew);
        ss[r] = scale;
        sl[r] = sl[r] * scale + psum;
        sm[r] = mnew;
      }
    }
    __syncthreads();
    // ---- O = O * scale + P V ----
    const float* vb = sv + buf * CA_KT * D;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float f = ss[4 * ty + a];
#pragma unroll
      for (int b = 0; b < 8; ++b) acc[a][b] *= f;
    }
#pragma unroll 4
    for (int s4 = 0; s4 < CA_KT / 4; ++s4) {
      float4 pa[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) pa[a] = reinterpret_cast<const float4*>(sp + (4 * ty + a) * (CA_KT + 4))[s4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 v0 = reinterpret_cast<const float4*>(vb + (4 * s4 + u) * D)[2 * tx];
        const float4 v1 = reinterpret_cast<const float4*>(vb + (4 * s4 + u) * D)[2 * tx + 1];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float p = u == 0 ? pa[a].x : u == 1 ? pa[a].y : u == 2 ? pa[a].z : pa[a].w;
          acc[a][0] = fmaf(p, v0.x, acc[a][0]); acc[a][1] = fmaf(p, v0.y, acc[a][1]);
          acc[a][2] = fmaf(p, v0.z, acc[a][2]); acc[a][3] = fmaf(p, v0.w, acc[a][3]);
          acc[a][4] = fmaf(p, v1.x, acc[a][4]); acc[a][5] = fmaf(p, v1.y, acc[a][5]);
          acc[a][6] = fmaf(p, v1.z, acc[a][6]); acc[a][7] = fmaf(p, v1.w, acc[a][7]);
        }
      }
    }
    __syncthreads();  // the buffer and P are reused by the next tile
  }
  // ---- output: normalised rows (one split) or row partials ----
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int r = 4 * ty + a;
    const int qi = qb0 + r / G, j = h * G + r % G;
    if (qi >= n_qpos) continue;
    const size_t row = (size_t)qi * hq + j;
    if (split == 1) {
      const float inv = sl[r] > 0.f ? 1.f / sl[r] : 0.f;
      float4* dst = reinterpret_cast<float4*>(o + row * D) + 2 * tx;
      dst[0] = make_float4(acc[a][0] * inv, acc[a][1] * inv, acc[a][2] * inv, acc[a][3] * inv);
      dst[1] = make_float4(acc[a][4] * inv, acc[a][5] * inv, acc[a][6] * inv, acc[a][7] * inv);
    } else {
      float* pp = part + ((size_t)sidx * n_qpos * hq + row) * (D + 4);
      float4* dst = reinterpret_cast<float4*>(pp) + 2 * tx;
      dst[0] = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      dst[1] = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
      if (tx == 0) {
        pp[D] = sm[r];
        pp[D + 1] = sl[r];
      }
    }
  }
}

// Log-sum-exp merge of the split partials of calib_attn_tiled_kernel, in split
// order.  One warp per (query position, query head); lane l: channels 4l..4l+3.
__global__ void calib_attn_combine_kernel(int n_rows, int split, const float* __restrict__ part,
                                          float* __restrict__ o) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  float M = -INFINITY;
  for (int s = 0; s < split; ++s) M = fmaxf(M, part[((size_t)s * n_rows + row) * (D + 4) + D]);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < split; ++s) {
      const float* pp = part + ((size_t)s * n_rows + row) * (D + 4);
      const float m = pp[D];
      if (m == -INFINITY) continue;
      const float e = __expf(m - M);
      const float4 x = reinterpret_cast<const float4*>(pp)[lane];
      L = fmaf(e, pp[D + 1], L);
      a.x = fmaf(e, x.x, a.x); a.y = fmaf(e, x.y, a.y); a.z = fmaf(e, x.z, a.z); a.w = fmaf(e, x.w, a.w);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  reinterpret_cast<float4*>(o + (size_t)row * D)[lane] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
}

template <int G>
static cudaError_t launch_calib_attn_g(int n_tok, int n_qpos, int n_kv_heads, const float* q, const float* k,
                                       const float* v, float* o, float* part, cudaStream_t s) {
  static std::atomic<unsigned long long> attr{0};  // per device
  const cudaError_t ea = smem_limit_once(attr, calib_attn_tiled_kernel<G>, CA_SMEM);
  if (ea != cudaSuccess) return ea;
  constexpr int QB = CA_ROWS / G;
  const int nqb = (n_qpos + QB - 1) / QB;
  const int n_tiles = (n_tok + CA_KT - 1) / CA_KT;
  int split = 152 / (n_kv_heads * nqb);  // about one CTA per SM
  if (split > CA_SPLIT_MAX) split = CA_SPLIT_MAX;
  if (split > n_tiles) split = n_tiles;
  if (split < 1) split = 1;
  calib_attn_tiled_kernel<G><<<dim3(n_kv_heads, nqb, split), 256, CA_SMEM, s>>>(n_tok, n_qpos, n_kv_heads, split, q, k,
                                                                                 v, o, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || split == 1) return e;
  const int rows = n_qpos * n_kv_heads * G;
  calib_attn_combine_kernel<<<(rows + 7) / 8, 256, 0, s>>>(rows, split, part, o);
  return cudaGetLastError();
}

static cudaError_t launch_calib_attn(int n_tok, int n_qpos, int n_kv_heads, int gqa, const float* q, const float* k,
                                     const float* v, float* o, float* part, cudaStream_t s) {
  switch (gqa) {
    case 1: return launch_calib_attn_g<1>(n_tok, n_qpos, n_kv_heads, q, k, v, o, part, s);
    case 2: return launch_calib_attn_g<2>(n_tok, n_qpos, n_kv_heads, q, k, v, o, part, s);
    case 4: return launch_calib_attn_g<4>(n_tok, n_qpos, n_kv_heads, q, k, v, o, part, s);
    case 8: return launch_calib_attn_g<8>(n_tok, n_qpos, n_kv_heads, q, k, v, o, part, s);
    default: return cudaErrorInvalidValue;
  }
}

// Gram matrices G_g = W_g^T W_g for head groups g of gd = cols columns each.
// w: [d_model][n_groups * gd]; gram: [n_groups][gd][gd].  32x32 tiles.
// Gram blocks G_g = W_g^T W_g (gd x gd) of the W_O columns of each scored group g:
// a block takes a 64 x 64 tile (thread: 4 x 4), K = d_model in chunks of 32 rows of W
// staged in shared memory as fp32.  grid = (gd / 64, gd / 64, n_groups), block = 256.
constexpr int GR_T = 64, GR_K = 32;
__global__ void __launch_bounds__(256) gram_kernel(int d_model, int total_cols, int gd,
                                                   const void* __restrict__ w, int w_dtype,
                                                   float* __restrict__ gram) {
  __shared__ __align__(16) float A[GR_K][GR_T + 4], B[GR_K][GR_T + 4];
  const int grp = blockIdx.z;
  const int a0 = blockIdx.y * GR_T, b0 = blockIdx.x * GR_T;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const size_t col0 = (size_t)grp * gd;
  // the next chunk's elements are loaded into registers while the current one is multiplied
  // thread: row tid / 8 of the chunk, columns 8 (tid % 8) .. + 7 of both tiles
  static_assert(GR_K * GR_T == 256 * 8, "one row segment of 8 columns per thread and tile");
  const int fr = tid >> 3, fc = 8 * (tid & 7);
  float4 na[2], nb[2];
  auto fetch = [&](int n0) {
    const int n = n0 + fr;
    const size_t row = (size_t)n * total_cols + col0;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    na[0] = n < d_model ? load4(w, row + a0 + fc, w_dtype) : z;
    na[1] = n < d_model ? load4(w, row + a0 + fc + 4, w_dtype) : z;
    nb[0] = n < d_model ? load4(w, row + b0 + fc, w_dtype) : z;
    nb[1] = n < d_model ? load4(w, row + b0 + fc + 4, w_dtype) : z;
  };
  fetch(0);
  for (int n0 = 0; n0 < d_model; n0 += GR_K) {
    *reinterpret_cast<float4*>(&A[fr][fc]) = na[0];
    *reinterpret_cast<float4*>(&A[fr][fc + 4]) = na[1];
    *reinterpret_cast<float4*>(&B[fr][fc]) = nb[0];
    *reinterpret_cast<float4*>(&B[fr][fc + 4]) = nb[1];
    __syncthreads();
    if (n0 + GR_K < d_model) fetch(n0 + GR_K);
#pragma unroll 8
    for (int r = 0; r < GR_K; ++r) {
      const float4 av = *reinterpret_cast<const float4*>(&A[r][4 * ty]);
      const float4 bv = *reinterpret_cast<const float4*>(&B[r][4 * tx]);
      const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(gram + ((size_t)grp * gd + a0 + 4 * ty + i) * gd + b0 + 4 * tx) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}

// trace(M du^T du) = sum_p du_p M du_p^T for one group (M = W_h^T W_h symmetric), as
// sum_{p,c} du[p][c] Z[p][c] with Z = du M: a block takes 64 columns of Z and a K range
// of `kspan` channels (both linear in Z, so ranges add), streams du[:, k] and M[k][c] through
// shared memory 64 x 64 at a time, and dots its Z tile with du[:, c] in double.
// grid = (gd / 64, ceil(gd / kspan), n_groups), block = 256 (thread: 4 x 4 of the tile).
constexpr int GT_T = 64;
__global__ void __launch_bounds__(256) gram_trace_kernel(int n_qpos, int n_groups, int gd, int kspan,
                                                         const float* __restrict__ a,
                                                         const float* __restrict__ b,
                                                         const float* __restrict__ gram,
                                                         double* __restrict__ part) {
  __shared__ float sdu[GT_T][GT_T + 1];  // du[p0 + p][k0 + k]
  __shared__ __align__(16) float smat[GT_T][GT_T + 4];  // M[k0 + k][c0 + c]
  __shared__ double sred[8];
  const int ct = blockIdx.x, ks = blockIdx.y, grp = blockIdx.z, tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int c0 = GT_T * ct, kb0 = ks * kspan, kb1 = min(gd, kb0 + kspan);
  const float* mg = gram + (size_t)grp * gd * gd;
  auto du_at = [&](int p, int k) {
    const size_t i = ((size_t)p * n_groups + grp) * gd + k;
    return b ? a[i] - b[i] : a[i];
  };
  double acc = 0.0;
  for (int p0 = 0; p0 < n_qpos; p0 += GT_T) {
    float z[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) z[i][j] = 0.f;
    for (int k0 = kb0; k0 < kb1; k0 += GT_T) {
      for (int i = tid; i < GT_T * GT_T; i += 256) {
        const int r = i >> 6, k = i & 63;
        sdu[r][k] = (p0 + r < n_qpos && k0 + k < kb1) ? du_at(p0 + r, k0 + k) : 0.f;
        smat[r][k] = k0 + r < kb1 ? mg[(size_t)(k0 + r) * gd + c0 + k] : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int k = 0; k < GT_T; ++k) {
        const float4 m4 = *reinterpret_cast<const float4*>(&smat[k][4 * tx]);
        const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float d = sdu[4 * ty + i][k];
#pragma unroll
          for (int j = 0; j < 4; ++j) z[i][j] = fmaf(d, mv[j], z[i][j]);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = p0 + 4 * ty + i;
      if (p < n_qpos)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc += (double)z[i][j] * (double)du_at(p, c0 + 4 * tx + j);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((tid & 31) == 0) sred[tid >> 5] = acc;
  __syncthreads();
  if (tid == 0) {
    double t = 0.0;
    for (int i = 0; i < 8; ++i) t += sred[i];
    part[((size_t)grp * gridDim.y + ks) * gridDim.x + ct] = t;
  }
}

// K span of the trace blocks: about two blocks per SM over all groups, at least 64 channels.
static int gram_kspan(int gd, int n_groups) {
  const int tiles = gd / GT_T;
  int ksplit = (2 * device_sm_count() + tiles * n_groups - 1) / (tiles * n_groups);
  ksplit = std::max(1, std::min(ksplit, gd / GT_T));
  return ((gd + ksplit - 1) / ksplit + GT_T - 1) / GT_T * GT_T;
}

__global__ void __launch_bounds__(256) gram_reduce_kernel(int n_tiles, const double* __restrict__ part,
                                                          double* __restrict__ out) {
  __shared__ double sh[256];
  const int g = blockIdx.x, tid = threadIdx.x;
  double t = 0.0;
  for (int i = tid; i < n_tiles; i += 256) t += part[(size_t)g * n_tiles + i];
  sh[tid] = t;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (tid < w) sh[tid] += sh[tid + w];
    __syncthreads();
  }
  if (tid == 0) out[g] = sh[0];
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
                         double* ref, void* ws, unsigned* err, cudaStream_t s) {
  const int hq = n_kv_heads * gqa;
  const int n_groups = calib_groups(n_kv_heads, joint);
  const int gd = calib_gd(n_kv_heads, gqa, joint);
  CalibWs w = carve(ws, n_tok, n_qpos, n_kv_heads, gqa, n_groups, gd, nullptr);
  const size_t qn = (size_t)n_qpos * hq * D, kn = (size_t)n_tok * n_kv_heads * D;
  auto blocks = [](size_t n) { return (unsigned)((n + 255) / 256); };

  to_f32_kernel<<<blocks(qn), 256, 0, s>>>(qn, hq, q, dtype, nullptr, w.qf);
  to_f32_kernel<<<blocks(kn), 256, 0, s>>>(kn, n_kv_heads, k, dtype, nullptr, w.kf);
  to_f32_kernel<<<blocks(kn), 256, 0, s>>>(kn, n_kv_heads, v, dtype, nullptr, w.vf);
  KVQ_TRY(cudaSuccess);
  // reference readout with unquantized, unrotated, uncentred keys and values
  KVQ_TRY(launch_calib_attn(n_tok, n_qpos, n_kv_heads, gqa, w.qf, w.kf, w.vf, w.o_ref, w.part, s));
  // ||du W^T||^2: directly when d_model <= gd, else through the group's Gram matrix
  const bool direct = d_model <= gd;
  if (!direct)
    gram_kernel<<<dim3(gd / GR_T, gd / GR_T, n_groups), 256, 0, s>>>(d_model, hq * D, gd, w_o, w_dtype, w.gram);
  zero_f64_kernel<<<1, 256, 0, s>>>(ref, n_groups);
  const int n_out = n_cand * n_clip * n_groups;
  zero_f64_kernel<<<(n_out + 255) / 256, 256, 0, s>>>(nmse, n_out);
  KVQ_TRY(cudaSuccess);
  const size_t form_smem = (size_t)gd * sizeof(float);
  auto out_err = [&](const float* a, const float* b, double* dst) {
    if (direct)
      proj_err_kernel<<<dim3(n_qpos, n_groups), 256, form_smem, s>>>(n_qpos, n_groups, gd, d_model, a, b, w_o,
                                                                     w_dtype, dst);
    else {
      const int ksp = gram_kspan(gd, n_groups), nks = (gd + ksp - 1) / ksp;
      gram_trace_kernel<<<dim3(gd / GT_T, nks, n_groups), 256, 0, s>>>(n_qpos, n_groups, gd, ksp, a, b, w.gram,
                                                                       w.gpart);
      gram_reduce_kernel<<<n_groups, 256, 0, s>>>((gd / GT_T) * nks, w.gpart, dst);
    }
  };
  out_err(w.o_ref, nullptr, ref);
  KVQ_TRY(cudaSuccess);
  // the quantized trace is read by the decode kernels: pages of CALIB_PAGE tokens, one
  // decode "sequence" per calibration position (its causal prefix), all sharing the pages
  const int n_blk = (n_tok + CALIB_PAGE - 1) / CALIB_PAGE;
  const PageGeom pg{CALIB_PAGE, n_kv_heads, n_blk, n_blk, 72 * CALIB_PAGE};
  KVQ_TRY(cudaMemsetAsync(w.pool, 0, (size_t)n_blk * n_kv_heads * 72 * CALIB_PAGE, s));
  calib_pages_kernel<<<(unsigned)(((long long)n_qpos * n_blk + 255) / 256), 256, 0, s>>>(n_qpos, n_tok, n_blk, w.table,
                                                                                        w.lens);
  KVQ_TRY(cudaSuccess);
  for (int i = 0; i < n_cand; ++i) {
    const RotDev r = to_dev(cand[i]);
    // keys centred (OptR §4.1; attention-equivalent) then rotated, values rotated: (k - mu) R
    // in double-float, so the decisions are those of the exact centred values
    KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, k, dtype, mu, r, w.xk_hi, w.xk_lo, s));
    KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, v, dtype, nullptr, r, w.xv_hi, w.xv_lo, s));
    for (int c = 0; c < n_clip; ++c) {
      // exact group decisions into the pool, then the decode of every prefix with the
      // candidate's query rotation (the cache path's own kernels: tensor-core contractions
      // on the 2-bit codes); o_rot in the rotated value basis
      KVQ_TRY(launch_quant_to_pool(n_tok, n_kv_heads, w.xk_hi, w.xk_lo, clips[c], 0, w.pool, s));
      KVQ_TRY(launch_quant_to_pool(n_tok, n_kv_heads, w.xv_hi, w.xv_lo, clips[c], 1, w.pool, s));
      KVQ_TRY(launch_decode(pg, hq, n_qpos, w.qf, KVQ_F32, w.lens, n_tok, w.table, r, w.pool, w.n_ctas, w.dws, w.o_rot,
                            err, s));
      KVQ_TRY(launch_rotate_heads(n_qpos, hq, gqa, w.o_rot, r, w.o_un, true, s));
      double* slot = nmse + (size_t)(i * n_clip + c) * n_groups;
      out_err(w.o_un, w.o_ref, slot);
      KVQ_TRY(cudaSuccess);
    }
  }
  divide_kernel<<<(n_out + 255) / 256, 256, 0, s>>>(nmse, ref, n_out, n_groups);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-head output-error report ("Output-Aware Rotation for INT2 KV-Cache
// Quantization", Figure 5 and the appendix "Output-space error"; Eq. 8).  Every
// query head j is scored on its own: ||Delta y_{t,j}||^2 = ||du W_O,j^T||^2 with
// du over the 128 channels of head j (groups of one query head).  Four causal
// attention passes over the trace:
//   reference  o   = softmax(q k) v                       raw keys and values
//   candidate  o~  = softmax(qR_K Q(kR_K)) Q(vR_V) R_V^T  (keys centred by mu)
//   keys only  o^K = softmax(qR_K Q(kR_K)) v              p~ with the exact values
//   plain INT2 o^N = softmax(q Q(k)) Q(v)                 identity, no centring
// give E = |o~ - o|, E_key = |o^K - o| (Eq. 8's (p~ - p) V term), E_val =
// |o~ - o^K| (its p~ (V~ - V) term), E_naive = |o^N - o| and Y = |o| (each the
// sum over positions of the squared post-W_O norms), summed per KV head.
// ---------------------------------------------------------------------------
__global__ void group_sum_kernel(int n_rows, int n_groups, int per, const double* __restrict__ in,
                                 double* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * n_groups) return;
  const int r = i / n_groups, g = i % n_groups;
  double t = 0.0;
  for (int j = 0; j < per; ++j) t += in[(size_t)r * n_groups * per + g * per + j];  // fixed order
  out[i] = t;
}

cudaError_t launch_head_report(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model, const void* q,
                               const void* k, const void* v, int dtype, const void* w_o, int w_dtype, RotDev rot_k,
                               RotDev rot_v, const float* mu, float clip_k, float clip_v, double* out, void* ws,
                               unsigned* err, cudaStream_t s) {
  const int hq = n_kv_heads * gqa;
  const int n_groups = hq, gd = D;
  CalibWs w = carve(ws, n_tok, n_qpos, n_kv_heads, gqa, n_groups, gd, nullptr);
  const size_t qn = (size_t)n_qpos * hq * D, kn = (size_t)n_tok * n_kv_heads * D;
  auto blocks = [](size_t n) { return (unsigned)((n + 255) / 256); };
  const RotDev ident{KVQ_ROT_IDENTITY, nullptr, nullptr};

  to_f32_kernel<<<blocks(qn), 256, 0, s>>>(qn, hq, q, dtype, nullptr, w.qf);
  to_f32_kernel<<<blocks(kn), 256, 0, s>>>(kn, n_kv_heads, k, dtype, nullptr, w.kf);
  to_f32_kernel<<<blocks(kn), 256, 0, s>>>(kn, n_kv_heads, v, dtype, nullptr, w.vf);
  zero_f64_kernel<<<1, 256, 0, s>>>(w.qsum, 5 * hq);
  KVQ_TRY(cudaSuccess);
  const bool direct = d_model <= gd;
  if (!direct)
    gram_kernel<<<dim3(gd / GR_T, gd / GR_T, n_groups), 256, 0, s>>>(d_model, hq * D, gd, w_o, w_dtype, w.gram);
  auto out_err = [&](const float* a, const float* b, double* dst) {
    if (direct)
      proj_err_kernel<<<dim3(n_qpos, n_groups), 256, (size_t)gd * sizeof(float), s>>>(n_qpos, n_groups, gd, d_model,
                                                                                   a, b, w_o, w_dtype, dst);
    else {
      const int ksp = gram_kspan(gd, n_groups), nks = (gd + ksp - 1) / ksp;
      gram_trace_kernel<<<dim3(gd / GT_T, nks, n_groups), 256, 0, s>>>(n_qpos, n_groups, gd, ksp, a, b, w.gram,
                                                                       w.gpart);
      gram_reduce_kernel<<<n_groups, 256, 0, s>>>((gd / GT_T) * nks, w.gpart, dst);
    }
  };
  double* e_tot = w.qsum;
  double* e_key = w.qsum + hq;
  double* e_val = w.qsum + 2 * hq;
  double* e_naive = w.qsum + 3 * hq;
  double* y_ref = w.qsum + 4 * hq;
  // the passes with INT2 keys and values read a page pool of the quantized trace with the
  // decode kernels (one sequence per position, as in the sweep)
  const int n_blk = (n_tok + CALIB_PAGE - 1) / CALIB_PAGE;
  const PageGeom pg{CALIB_PAGE, n_kv_heads, n_blk, n_blk, 72 * CALIB_PAGE};
  KVQ_TRY(cudaMemsetAsync(w.pool, 0, (size_t)n_blk * n_kv_heads * 72 * CALIB_PAGE, s));
  calib_pages_kernel<<<(unsigned)(((long long)n_qpos * n_blk + 255) / 256), 256, 0, s>>>(n_qpos, n_tok, n_blk, w.table,
                                                                                        w.lens);
  KVQ_TRY(cudaSuccess);
  // reference
  KVQ_TRY(launch_calib_attn(n_tok, n_qpos, n_kv_heads, gqa, w.qf, w.kf, w.vf, w.o_ref, w.part, s));
  out_err(w.o_ref, nullptr, y_ref);
  // candidate: keys centred and rotated by R_K, values rotated by R_V, both INT2
  KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, k, dtype, mu, rot_k, w.xk_hi, w.xk_lo, s));
  KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, v, dtype, nullptr, rot_v, w.xv_hi, w.xv_lo, s));
  KVQ_TRY(launch_quant_to_pool(n_tok, n_kv_heads, w.xk_hi, w.xk_lo, clip_k, 0, w.pool, s));
  KVQ_TRY(launch_quant_to_pool(n_tok, n_kv_heads, w.xv_hi, w.xv_lo, clip_v, 1, w.pool, s));
  KVQ_TRY(launch_decode(pg, hq, n_qpos, w.qf, KVQ_F32, w.lens, n_tok, w.table, rot_k, w.pool, w.n_ctas, w.dws,
                        w.o_rot, err, s));
  KVQ_TRY(launch_rotate_heads(n_qpos, hq, gqa, w.o_rot, rot_v, w.o_un, true, s));  // o~ (unrotated)
  out_err(w.o_un, w.o_ref, e_tot);
  KVQ_TRY(launch_rotate_heads(n_qpos, hq, gqa, w.qf, rot_k, w.qr, false, s));
  KVQ_TRY(launch_quant_dequant(n_tok * n_kv_heads, w.xk_hi, w.xk_lo, clip_k, w.kq, s));
  // keys only: the candidate's weights p~ with the exact values (unrotated basis)
  KVQ_TRY(launch_calib_attn(n_tok, n_qpos, n_kv_heads, gqa, w.qr, w.kq, w.vf, w.o_rot, w.part, s));
  out_err(w.o_rot, w.o_ref, e_key);
  out_err(w.o_un, w.o_rot, e_val);
  // plain per-group INT2: identity rotations, no centring, the same clips
  KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, k, dtype, nullptr, ident, w.xk_hi, w.xk_lo, s));
  KVQ_TRY(launch_rotate_df(n_tok, n_kv_heads, v, dtype, nullptr, ident, w.xv_hi, w.xv_lo, s));
  KVQ_TRY(launch_quant_to_pool(n_tok, n_kv_heads, w.xk_hi, w.xk_lo, clip_k, 0, w.pool, s));
  KVQ_TRY(launch_quant_to_pool(n_tok, n_kv_heads, w.xv_hi, w.xv_lo, clip_v, 1, w.pool, s));
  KVQ_TRY(launch_decode(pg, hq, n_qpos, w.qf, KVQ_F32, w.lens, n_tok, w.table, ident, w.pool, w.n_ctas, w.dws,
                        w.o_rot, err, s));
  out_err(w.o_rot, w.o_ref, e_naive);
  group_sum_kernel<<<blocks(5 * n_kv_heads), 256, 0, s>>>(5, n_kv_heads, gqa, w.qsum, out);
  return cudaGetLastError();
}

}  // namespace kvq
