// Read path: split-K decode attention straight off the packed INT2 pages, and
// the log-sum-exp combine of the split partials.
//
// "Output-Aware Rotation for INT2 KV-Cache Quantization": Eqs. 1-2 and 5
// (logits <q, k~>/sqrt(d), softmax over the cached positions, o = p^T V~),
// appendix Eqs. 21-22 / 26 (the query is rotated once, q R_K, and meets the
// stored rotated keys), Eq. 27 (the readout stays in the rotated-V basis).
// Scale and zero are factored out of the dot products, which is exact algebra:
//   q'.(z + s c) = s (q'.c) + z sum(q'),    sum_t p_t (z_t + s_t c_t) = sum_t (p_t s_t) c_t + sum_t p_t z_t.
// The softmax runs in base 2 (q' is pre-scaled by log2(e)/sqrt(128)).
#include "quant_common.cuh"

namespace kvq {

constexpr float LOG2E = 1.4426950408889634f;

// Per-CTA partial: acc[B][Hq][S][128], then ml[B][Hq][S][2] (running max m in
// log2 units, sum l).
struct Partials {
  float* acc;
  float* ml;
};

__host__ __device__ inline Partials partials_from_ws(void* ws, int n_seqs, int n_q_heads, int n_splits) {
  Partials p;
  p.acc = static_cast<float*>(ws);
  p.ml = p.acc + (size_t)n_seqs * n_q_heads * n_splits * D;
  return p;
}

size_t decode_workspace_bytes(int n_seqs, int n_q_heads, int n_splits) {
  return (size_t)n_seqs * n_q_heads * n_splits * (D + 2) * sizeof(float);
}

int decode_auto_splits(int n_seqs, int n_kv_heads, int max_seq_len, int page_tokens) {
  int pages = (max_seq_len + page_tokens - 1) / page_tokens;
  long long units = (long long)n_seqs * n_kv_heads;
  int target = 152 * 4;
  int s = (int)((target + units - 1) / units);
  int cap = pages / 16 > 1 ? pages / 16 : 1;  // keep >= 16 pages per split
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  if (s > 256) s = 256;
  return s;
}

// grid = (n_splits, n_kv_heads, n_seqs), block = 128 (4 warps).  Each warp walks
// the split's pages round robin with its own online-softmax state; the four
// states are merged in shared memory at the end.
template <int G, int P>
__global__ void __launch_bounds__(128) decode_split_kernel(
    PageGeom g, int n_q_heads, const void* __restrict__ q, int q_dtype,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ table, RotDev rot_k,
    const uint8_t* __restrict__ pool, int n_splits, Partials part, unsigned* err) {
  constexpr int LPT = 32 / P;      // lanes per token in the score phase
  constexpr int CPL = D / LPT;     // channels per lane in the score phase
  constexpr int KOFF = 0, VOFF = 32 * P, KMETA = 64 * P, VMETA = 68 * P;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  __shared__ __align__(16) float qs[G][D];
  __shared__ float qsum[G];
  __shared__ float sm_m[4][G], sm_l[4][G];
  __shared__ __align__(16) float sm_acc[4][G][D];

  // Prologue: q'_j = q_j R_K,h scaled by log2(e)/sqrt(128) (Eq. 22).
  for (int jj = warp; jj < G; jj += 4) {
    const int j = h * G + jj;
    float4 v = load4(q, ((size_t)b * n_q_heads + j) * D + 4 * lane, q_dtype);
    v = rotate_vec_warp(v, rot_k, h, lane, false);
    const float sc = LOG2E * INV_SQRT_D;
    v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
    reinterpret_cast<float4*>(qs[jj])[lane] = v;
    float tot = warp_sum(v.x + v.y + v.z + v.w);
    if (lane == 0) qsum[jj] = tot;
  }
  __syncthreads();

  int len = __ldg(seq_lens + b);
  if (len < 0 || len > g.max_blocks * g.page_tokens) {
    if (threadIdx.x == 0) flag_error(err, ERR_SEQ_RANGE);
    len = 0;
  }
  const int n_pages = (len + P - 1) / P;
  const int pps = (n_pages + n_splits - 1) / n_splits;
  const int p_begin = split * pps;
  const int p_end = min(n_pages, p_begin + pps);

  float m[G], l[G];
  float4 acc[G];
#pragma unroll
  for (int j = 0; j < G; ++j) { m[j] = -INFINITY; l[j] = 0.f; acc[j] = make_float4(0.f, 0.f, 0.f, 0.f); }

  const int tok = lane / LPT;        // score phase: token handled by this lane
  const int sub = lane % LPT;        // which CPL-channel slice
  for (int p = p_begin + warp; p < p_end; p += 4) {
    const int blk = __ldg(table + (size_t)b * g.max_blocks + p);
    if (blk < 0 || blk >= g.num_blocks) {
      if (lane == 0) flag_error(err, ERR_BLOCK_RANGE);
      continue;
    }
    const uint8_t* rec = pool + ((size_t)blk * g.n_kv_heads + h) * g.record;
    const int nv = min(P, len - p * P);

    // ---- scores: lane covers token `tok`, channels [sub*CPL, (sub+1)*CPL) ----
    float dot[G];
#pragma unroll
    for (int j = 0; j < G; ++j) dot[j] = 0.f;
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(rec + KOFF + 32 * tok + (CPL / 4) * sub);
#pragma unroll
    for (int wi = 0; wi < CPL / 16; ++wi) {
      const uint32_t w = __ldg(kw + wi);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float c = (float)((w >> (2 * i)) & 3u);
        const int ch = sub * CPL + wi * 16 + i;
#pragma unroll
        for (int j = 0; j < G; ++j) dot[j] = fmaf(c, qs[j][ch], dot[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
      for (int o = 1; o < LPT; o <<= 1) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], o);
    }
    const uint32_t km = __ldg(reinterpret_cast<const uint32_t*>(rec + KMETA + 4 * tok));
    const float ks = __half2float(__ushort_as_half((unsigned short)(km & 0xFFFFu)));
    const float kz = __half2float(__ushort_as_half((unsigned short)(km >> 16)));
    float sc[G], pr[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      sc[j] = tok < nv ? fmaf(ks, dot[j], kz * qsum[j]) : -INFINITY;
      float mp = sc[j];
#pragma unroll
      for (int o = LPT; o < 32; o <<= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
      const float mnew = fmaxf(m[j], mp);
      const float alpha = exp2f(m[j] - mnew);
      pr[j] = exp2f(sc[j] - mnew);
      float ps = pr[j];
#pragma unroll
      for (int o = LPT; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[j] = l[j] * alpha + ps;
      m[j] = mnew;
      acc[j].x *= alpha; acc[j].y *= alpha; acc[j].z *= alpha; acc[j].w *= alpha;
    }

    // ---- values: lane owns channels 4*lane .. 4*lane+3 (byte `lane` of each V row) ----
    for (int t = 0; t < nv; ++t) {
      const uint32_t vb = rec[VOFF + 32 * t + lane];
      const uint32_t vm = __ldg(reinterpret_cast<const uint32_t*>(rec + VMETA + 4 * t));
      const float vs = __half2float(__ushort_as_half((unsigned short)(vm & 0xFFFFu)));
      const float vz = __half2float(__ushort_as_half((unsigned short)(vm >> 16)));
      const float v0 = fmaf(vs, (float)(vb & 3u), vz), v1 = fmaf(vs, (float)((vb >> 2) & 3u), vz);
      const float v2 = fmaf(vs, (float)((vb >> 4) & 3u), vz), v3 = fmaf(vs, (float)((vb >> 6) & 3u), vz);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float pt = __shfl_sync(0xffffffffu, pr[j], t * LPT);
        acc[j].x = fmaf(pt, v0, acc[j].x); acc[j].y = fmaf(pt, v1, acc[j].y);
        acc[j].z = fmaf(pt, v2, acc[j].z); acc[j].w = fmaf(pt, v3, acc[j].w);
      }
    }
  }

  // ---- merge the four warps' states ----
#pragma unroll
  for (int j = 0; j < G; ++j) {
    if (lane == 0) { sm_m[warp][j] = m[j]; sm_l[warp][j] = l[j]; }
    reinterpret_cast<float4*>(sm_acc[warp][j])[lane] = acc[j];
  }
  __syncthreads();
  const int c = threadIdx.x;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float M = fmaxf(fmaxf(sm_m[0][j], sm_m[1][j]), fmaxf(sm_m[2][j], sm_m[3][j]));
    float A = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float e = exp2f(sm_m[w][j] - M);
        A = fmaf(e, sm_acc[w][j][c], A);
        L = fmaf(e, sm_l[w][j], L);
      }
    }
    const size_t row = ((size_t)b * n_q_heads + h * G + j) * n_splits + split;
    part.acc[row * D + c] = A;
    if (c == 0) { part.ml[row * 2] = M; part.ml[row * 2 + 1] = L; }
  }
}

// grid = (n_q_heads, n_seqs), block = 128: o = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
__global__ void __launch_bounds__(128) decode_combine_kernel(int n_q_heads, int n_splits,
                                                             Partials part, float* __restrict__ o) {
  const int j = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const size_t base = ((size_t)b * n_q_heads + j) * n_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part.ml[(base + s) * 2]);
  float A = 0.f, L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float e = exp2f(part.ml[(base + s) * 2] - M);
      L = fmaf(e, part.ml[(base + s) * 2 + 1], L);
      A = fmaf(e, part.acc[(base + s) * D + c], A);
    }
  }
  o[((size_t)b * n_q_heads + j) * D + c] = L > 0.f ? A / L : 0.f;
}

cudaError_t launch_decode(const PageGeom& g, int n_q_heads, int n_seqs, const void* q,
                          int q_dtype, const int32_t* seq_lens, int max_seq_len,
                          const int32_t* table, RotDev rot_k, const uint8_t* pool, int n_splits,
                          void* ws, float* o_rot, unsigned* err, cudaStream_t s) {
  if (n_seqs == 0) return cudaSuccess;
  const int gqa = n_q_heads / g.n_kv_heads;
  Partials part = partials_from_ws(ws, n_seqs, n_q_heads, n_splits);
  dim3 grid(n_splits, g.n_kv_heads, n_seqs);
#define KVQ_DEC(GG, PP) \
  decode_split_kernel<GG, PP><<<grid, 128, 0, s>>>(g, n_q_heads, q, q_dtype, seq_lens, table, rot_k, pool, n_splits, part, err)
#define KVQ_DEC_P(GG) \
  if (g.page_tokens == 16) KVQ_DEC(GG, 16); else KVQ_DEC(GG, 8)
  switch (gqa) {
    case 1: KVQ_DEC_P(1); break;
    case 2: KVQ_DEC_P(2); break;
    case 4: KVQ_DEC_P(4); break;
    case 8: KVQ_DEC_P(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_DEC_P
#undef KVQ_DEC
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(n_q_heads, n_seqs), 128, 0, s>>>(n_q_heads, n_splits, part, o_rot);
  return cudaGetLastError();
}

}  // namespace kvq
