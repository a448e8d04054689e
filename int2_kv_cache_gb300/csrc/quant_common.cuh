// Group quantizer shared by the write path and the calibration sweep.
//
// One group = the 128 channels of one token of one head ("Output-Aware Rotation
// for INT2 KV-Cache Quantization", §3.1 Eq. 4 and §5 implementation details:
// group-wise affine INT2, group size 128, clip ratio c; fp16 scale and zero as
// the 2.32 bits-per-element accounting implies):
//   lo = c * min(x), hi = c * max(x)
//   scale = fp16_rn((hi - lo) / 3), zero = fp16_rn(lo)
//   code  = clamp(round_half_even((x - zero) / scale), 0, 3), 0 where scale == 0
//
// Every decision that turns floating point into an integer (the fp16 rounding of
// scale and zero, the code of each channel) is taken on x carried as an unevaluated
// sum of two floats ("double-float", ~48 significant bits) and decided exactly:
// the fp16 roundings look at the low word at exact midpoints, and codes come from
// exact comparisons of x - zero with the rounding midpoints 0.5, 1.5 and 2.5 times
// scale.  The rotations that produce x carry their rounding errors the same way
// (compensated butterflies for the Walsh-Hadamard transform, error-free products
// and sums for dense matrices; Ogita, Rump & Oishi, "Accurate sum and dot
// product", 2005).  The result equals the decision on the exact real x except
// within ~1e-13 (relative) of a rounding boundary.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

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

// One role of a cache write (keys or values): input rows, rotation, rotated key
// mean (or nullptr), clip ratio and the offsets of its codes and meta in a record.
struct AppendRole {
  const void* src;
  RotDev rot;
  const float* mu_rot;
  float clip;
  int codes_off, meta_off;
};
struct AppendRoles {
  AppendRole r[2];
};

// Bulk cache write of dense roles on the tensor cores (append_tc.cu): roles.r[0 ..
// n_roles - 1] must be dense; inputs and pool 16-byte aligned (append_dense_tc_supported).
bool append_dense_tc_supported(int dtype, const void* k, const void* v, const uint8_t* pool);
cudaError_t launch_append_dense_tc(const PageGeom& g, int n_seqs, int n_new, int dtype, const int32_t* cu_new,
                                   const int32_t* start_pos, const int32_t* table, const AppendRoles& roles,
                                   int n_roles, uint8_t* pool, unsigned* err, cudaStream_t s);

// ---------------------------------------------------------------------------
// double-float arithmetic (intrinsics keep the compiler from fusing or reordering)
// ---------------------------------------------------------------------------
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return DF{s, e};
}

// Renormalise hi + lo (any magnitudes) so that |lo| <= ulp(hi) / 2.
__device__ __forceinline__ DF df_norm(float hi, float lo) { return two_sum(hi, lo); }

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  return df_norm(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ DF df_add_f(DF a, float b) {
  const DF s = two_sum(a.hi, b);
  return df_norm(s.hi, __fadd_rn(s.lo, a.lo));
}

__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const float p = __fmul_rn(a.hi, b);
  float e = __fmaf_rn(a.hi, b, -p);
  e = __fmaf_rn(a.lo, b, e);
  return df_norm(p, e);
}

// 1 / sqrt(128) as a double-float.
constexpr float INV_SQRT_D = 0.0883883461356163f;
constexpr float INV_SQRT_D_LO = 1.512702185735293e-09f;

__device__ __forceinline__ DF df_mul_inv_sqrt_d(DF a) {
  const float p = __fmul_rn(a.hi, INV_SQRT_D);
  float e = __fmaf_rn(a.hi, INV_SQRT_D, -p);
  e = __fmaf_rn(a.hi, INV_SQRT_D_LO, e);
  e = __fmaf_rn(a.lo, INV_SQRT_D, e);
  return df_norm(p, e);
}

__device__ __forceinline__ bool df_less(DF a, DF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

// fp16 rounding (to nearest, ties to even) of the exact value hi + lo.
__device__ __forceinline__ __half df_to_half(DF v) {
  __half h = __float2half_rn(v.hi);
  const float hf = __half2float(h);
  if (v.lo != 0.f && hf != v.hi && isfinite(hf)) {
    // v.hi was rounded to h; only if v.hi sits exactly on the midpoint between h
    // and its other neighbour can the low word change the result.
    const unsigned short hb = __half_as_ushort(h);
    const bool away = fabsf(v.hi) > fabsf(hf);  // v.hi lies further from zero than h
    const unsigned short nb = away ? (unsigned short)(hb + 1) : (unsigned short)(hb - 1);
    const float nf = __half2float(__ushort_as_half(nb));
    if (__fsub_rn(v.hi, hf) == __fsub_rn(nf, v.hi)) {
      const bool lo_toward_n = (nf > v.hi) == (v.lo > 0.f);
      if (lo_toward_n) h = __ushort_as_half(nb);
    }
  }
  return h;
}

struct QParams {
  unsigned short s_bits, z_bits;
  float s, z;           // fp16-rounded scale and zero (exact as float)
  float t05, t15, t25;  // rounding midpoints 0.5 s, 1.5 s, 2.5 s (exact in fp32)
};

// Scale and zero from the group's (double-float) min and max.
__device__ __forceinline__ QParams qparams_df(DF mn, DF mx, float clip) {
  const DF lo = df_mul_f(mn, clip);
  const DF hi = df_mul_f(mx, clip);
  const DF range = df_add(hi, DF{-lo.hi, -lo.lo});
  // range / 3 as a double-float: q = fl(range.hi / 3), remainder exact by FMA
  const float q = __fdiv_rn(range.hi, 3.0f);
  const float r = __fadd_rn(__fmaf_rn(-q, 3.0f, range.hi), range.lo);
  const DF third = df_norm(q, __fdiv_rn(r, 3.0f));
  const __half s16 = df_to_half(third);
  const __half z16 = df_to_half(lo);
  QParams p;
  p.s_bits = __half_as_ushort(s16);
  p.z_bits = __half_as_ushort(z16);
  p.s = __half2float(s16);
  p.z = __half2float(z16);
  p.t05 = 0.5f * p.s;
  p.t15 = 1.5f * p.s;
  p.t25 = 2.5f * p.s;
  return p;
}

// round_half_even((x - zero) / scale) clamped to [0, 3], decided exactly on x = hi + lo.
__device__ __forceinline__ unsigned qcode_df(DF x, const QParams& p) {
  if (!(p.s > 0.f)) return 0u;
  const DF d = df_add_f(x, -p.z);
  const unsigned a = (d.hi > p.t05 || (d.hi == p.t05 && d.lo > 0.f)) ? 1u : 0u;   // tie at .5 -> 0
  const unsigned b = (d.hi > p.t15 || (d.hi == p.t15 && d.lo >= 0.f)) ? 1u : 0u;  // tie at 1.5 -> 2
  const unsigned c = (d.hi > p.t25 || (d.hi == p.t25 && d.lo > 0.f)) ? 1u : 0u;   // tie at 2.5 -> 2
  return a + b + c;
}

// Paired fp32 arithmetic of sm_100 (two lanes of a 64-bit register per instruction).
__device__ __forceinline__ uint64_t f2pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2up(uint64_t p) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ---------------------------------------------------------------------------
// warp helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ DF shfl_xor_df(DF v, int m) {
  return DF{__shfl_xor_sync(0xffffffffu, v.hi, m), __shfl_xor_sync(0xffffffffu, v.lo, m)};
}

// min and max over the 128 double-float values of a warp (4 per lane).
__device__ __forceinline__ void warp_minmax_df(const DF x[4], DF& mn, DF& mx) {
  mn = x[0];
  mx = x[0];
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    if (df_less(x[i], mn)) mn = x[i];
    if (df_less(mx, x[i])) mx = x[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const DF a = shfl_xor_df(mn, o), b = shfl_xor_df(mx, o);
    if (df_less(a, mn)) mn = a;
    if (df_less(mx, b)) mx = b;
  }
}

// ---------------------------------------------------------------------------
// Rotations of one head vector held by a warp (lane l owns channels 4l..4l+3).
// ---------------------------------------------------------------------------

// Compensated Walsh-Hadamard transform (Sylvester order, unnormalised): every
// butterfly keeps its rounding error in the low word.
__device__ __forceinline__ DF df_bfly_add(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  return DF{s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo))};
}
__device__ __forceinline__ DF df_bfly_sub(DF a, DF b) {
  const DF s = two_sum(a.hi, -b.hi);
  return DF{s.hi, __fadd_rn(s.lo, __fsub_rn(a.lo, b.lo))};
}

__device__ __forceinline__ void warp_fwht128_df(DF v[4], int lane) {
  DF a0 = df_bfly_add(v[0], v[1]), a1 = df_bfly_sub(v[0], v[1]);
  DF a2 = df_bfly_add(v[2], v[3]), a3 = df_bfly_sub(v[2], v[3]);
  v[0] = df_bfly_add(a0, a2);
  v[2] = df_bfly_sub(a0, a2);
  v[1] = df_bfly_add(a1, a3);
  v[3] = df_bfly_sub(a1, a3);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const DF p = shfl_xor_df(v[i], m);
      v[i] = upper ? df_bfly_sub(p, v[i]) : df_bfly_add(v[i], p);
    }
  }
}

// x (4 channels per lane, double-float) -> x R_head as double-float.
//   signed Hadamard: R = diag(s) H / sqrt(128)
//   dense:           y_d = sum_c x_c R[c][d], error-free products and sums
__device__ __forceinline__ void rotate_df_warp(DF x[4], const RotDev& rot, int head, int lane) {
  if (rot.kind == KVQ_ROT_SIGNED_HADAMARD) {
    const float4 s = __ldg(reinterpret_cast<const float4*>(rot.signs + (size_t)head * D) + lane);
    x[0].hi *= s.x; x[0].lo *= s.x; x[1].hi *= s.y; x[1].lo *= s.y;
    x[2].hi *= s.z; x[2].lo *= s.z; x[3].hi *= s.w; x[3].lo *= s.w;
    warp_fwht128_df(x, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = df_mul_inv_sqrt_d(x[i]);
  } else if (rot.kind == KVQ_ROT_DENSE) {
    const float* R = rot.dense + (size_t)head * D * D;
    float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int c = 0; c < D; ++c) {
      const int src = c >> 2, k = c & 3;
      const float xh = __shfl_sync(0xffffffffu, k == 0 ? x[0].hi : k == 1 ? x[1].hi : k == 2 ? x[2].hi : x[3].hi, src);
      const float xl = __shfl_sync(0xffffffffu, k == 0 ? x[0].lo : k == 1 ? x[1].lo : k == 2 ? x[2].lo : x[3].lo, src);
      const float4 r4 = __ldg(reinterpret_cast<const float4*>(R + (size_t)c * D) + lane);
      const float r[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __fmul_rn(xh, r[i]);
        float pe = __fmaf_rn(xh, r[i], -p);
        pe = __fmaf_rn(xl, r[i], pe);
        const DF t = two_sum(sh[i], p);
        sh[i] = t.hi;
        sl[i] = __fadd_rn(sl[i], __fadd_rn(t.lo, pe));
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = df_norm(sh[i], sl[i]);
  }
}

// Plain fp32 rotation of a warp-held vector (query rotation and the inverse
// rotation of calibration readouts, which feed continuous outputs only):
// y = x R_head, or y = x R_head^T when `transpose`.
__device__ __forceinline__ float4 rotate_vec_warp(float4 v, const RotDev& rot, int head, int lane,
                                                  bool transpose) {
  if (rot.kind == KVQ_ROT_SIGNED_HADAMARD) {
    const float4 s = __ldg(reinterpret_cast<const float4*>(rot.signs + (size_t)head * D) + lane);
    if (!transpose) { v.x *= s.x; v.y *= s.y; v.z *= s.z; v.w *= s.w; }
    float a0 = v.x + v.y, a1 = v.x - v.y, a2 = v.z + v.w, a3 = v.z - v.w;
    v.x = a0 + a2; v.z = a0 - a2; v.y = a1 + a3; v.w = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float px = __shfl_xor_sync(0xffffffffu, v.x, m), py = __shfl_xor_sync(0xffffffffu, v.y, m);
      const float pz = __shfl_xor_sync(0xffffffffu, v.z, m), pw = __shfl_xor_sync(0xffffffffu, v.w, m);
      if (lane & m) { v.x = px - v.x; v.y = py - v.y; v.z = pz - v.z; v.w = pw - v.w; }
      else          { v.x = v.x + px; v.y = v.y + py; v.z = v.z + pz; v.w = v.w + pw; }
    }
    v.x *= INV_SQRT_D; v.y *= INV_SQRT_D; v.z *= INV_SQRT_D; v.w *= INV_SQRT_D;
    if (transpose) { v.x *= s.x; v.y *= s.y; v.z *= s.z; v.w *= s.w; }
    return v;
  }
  if (rot.kind == KVQ_ROT_DENSE) {
    const float* R = rot.dense + (size_t)head * D * D;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!transpose) {
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        const float src = (c & 3) == 0 ? v.x : (c & 3) == 1 ? v.y : (c & 3) == 2 ? v.z : v.w;
        const float xc = __shfl_sync(0xffffffffu, src, c >> 2);
        const float4 r = __ldg(reinterpret_cast<const float4*>(R + (size_t)c * D) + lane);
        y.x = fmaf(xc, r.x, y.x); y.y = fmaf(xc, r.y, y.y);
        y.z = fmaf(xc, r.z, y.z); y.w = fmaf(xc, r.w, y.w);
      }
    } else {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4* row = reinterpret_cast<const float4*>(R + (size_t)(4 * lane + i) * D);
        float part = 0.f;
        for (int c4 = 0; c4 < 32; ++c4) {
          const float4 r = __ldg(row + c4);
          const float x0 = __shfl_sync(0xffffffffu, v.x, c4), x1 = __shfl_sync(0xffffffffu, v.y, c4);
          const float x2 = __shfl_sync(0xffffffffu, v.z, c4), x3 = __shfl_sync(0xffffffffu, v.w, c4);
          part = fmaf(x0, r.x, part); part = fmaf(x1, r.y, part);
          part = fmaf(x2, r.z, part); part = fmaf(x3, r.w, part);
        }
        acc[i] = part;
      }
      y = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    return y;
  }
  return v;
}

// ---------------------------------------------------------------------------
// Certified fp32 path.  The group is first decided from fp32 values d_i that
// are known to lie within E of the exact x_i (E from an a-priori bound on the
// fp32 rotation and subtraction errors).  A decision (the fp16 rounding of
// scale or zero, a code) is taken only if no value in [d - E, d + E] could
// change it; it then equals the decision on the exact x, which is what the
// double-float path computes too.  Otherwise the caller falls back to the
// double-float path for the whole group.  Ties always fall back.
// ---------------------------------------------------------------------------

// Powers of two for the error bounds (exact multiplies).
constexpr float P2_M19 = 1.9073486328125e-06f;  // 2^-19
constexpr float P2_M22 = 2.384185791015625e-07f;  // 2^-22 = 4 u

// fp16 rounding of the exact value v* with |v* - v| <= err: true and h =
// fp16_rn(v*) when every value in that interval rounds alike (finite).
__device__ __forceinline__ bool half_rn_certain(float v, float err, __half& h) {
  err = __fmaf_rn(fabsf(v), P2_M22, err);  // covers the rounding of v - err and v + err
  const __half a = __float2half_rn(__fsub_rn(v, err)), b = __float2half_rn(__fadd_rn(v, err));
  h = a;
  return __half_as_ushort(a) == __half_as_ushort(b) && (__half_as_ushort(a) & 0x7c00u) != 0x7c00u;
}

// x R_head in fp32 for the identity and signed-Hadamard kinds (lane l holds
// channels 4l..4l+3; the input values are exact floats and the signs +-1).
// Returns B with |y_i - (x R)_i| <= B for every channel of the warp.
__device__ __forceinline__ float rotate_f32_bounded(float y[4], const RotDev& rot, int head, int lane) {
  if (rot.kind != KVQ_ROT_SIGNED_HADAMARD) return 0.f;  // identity: exact
  const float4 s = __ldg(reinterpret_cast<const float4*>(rot.signs + (size_t)head * D) + lane);
  y[0] *= s.x; y[1] *= s.y; y[2] *= s.z; y[3] *= s.w;
  // every butterfly stage adds at most u * sum|x| to each output (the nodes an
  // output depends on at one stage partition the inputs); 7 stages, then the
  // scaling by fp32(1/sqrt(128)) (relative error < 0.2 u) and its rounding
  const float l1 = warp_sum(fabsf(y[0]) + fabsf(y[1]) + fabsf(y[2]) + fabsf(y[3]));
  float a0 = y[0] + y[1], a1 = y[0] - y[1], a2 = y[2] + y[3], a3 = y[2] - y[3];
  y[0] = a0 + a2; y[2] = a0 - a2; y[1] = a1 + a3; y[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float sg = (lane & m) ? -1.f : 1.f;  // upper half: p - y, lower half: y + p
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = __shfl_xor_sync(0xffffffffu, y[i], m);
      y[i] = __fmaf_rn(sg, y[i], p);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = __fmul_rn(y[i], INV_SQRT_D);
  // 8.2 u * l1 / sqrt(128) + u |y|, with |y| <= l1 / sqrt(128), and a factor 2 of margin
  return l1 * INV_SQRT_D * P2_M19;
}

// Scale and zero of a group whose exact min and max lie within E of mn and mx:
// true when both fp16 roundings are certain (p then holds them, as qparams_df
// would compute them from the exact values); p is filled either way.
__device__ __forceinline__ bool qparams_certain(float mn, float mx, float E, float clip, QParams& p) {
  const float lo = __fmul_rn(clip, mn), hi = __fmul_rn(clip, mx);
  const float elo = __fmaf_rn(clip, E, fabsf(lo) * P2_M22);
  const float ehi = __fmaf_rn(clip, E, fabsf(hi) * P2_M22);
  const float range = __fsub_rn(hi, lo);
  const float third = __fdiv_rn(range, 3.0f);
  const float eth = (elo + ehi + fabsf(range) * P2_M22) * 0.3334f + fabsf(third) * P2_M22;
  __half s16, z16;
  bool ok = half_rn_certain(third, eth, s16);
  ok = half_rn_certain(lo, elo, z16) && ok;
  p.s_bits = __half_as_ushort(s16);
  p.z_bits = __half_as_ushort(z16);
  p.s = __half2float(s16);
  p.z = __half2float(z16);
  p.t05 = 0.5f * p.s;
  p.t15 = 1.5f * p.s;
  p.t25 = 2.5f * p.s;
  return ok;
}

// Code of d (|d - x| <= E) under p; `certain` is cleared when x could take another code.
__device__ __forceinline__ unsigned qcode_certain(float d, float E, const QParams& p, bool& certain) {
  const float dz = __fsub_rn(d, p.z);
  const float eb = __fmaf_rn(fabsf(d) + fabsf(dz), P2_M22, E);
  certain = fabsf(__fsub_rn(dz, p.t05)) > eb && fabsf(__fsub_rn(dz, p.t15)) > eb && fabsf(__fsub_rn(dz, p.t25)) > eb;
  return (dz > p.t05 ? 1u : 0u) + (dz > p.t15 ? 1u : 0u) + (dz > p.t25 ? 1u : 0u);
}

// Group decision from d (|d_i - x_i| <= E for every channel of the warp).
// Returns false (warp-uniform) when some decision is not certain.
__device__ __forceinline__ bool quantize_warp_certain(const float d[4], float E, float clip, QParams& p,
                                                      unsigned& byte) {
  const float mn = warp_min(fminf(fminf(d[0], d[1]), fminf(d[2], d[3])));
  const float mx = warp_max(fmaxf(fmaxf(d[0], d[1]), fmaxf(d[2], d[3])));
  // exact min / max lie within E of mn / mx
  bool ok = qparams_certain(mn, mx, E, clip, p);
  byte = 0u;
  if (p.s > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      bool c_ok;
      const unsigned c = qcode_certain(d[i], E, p, c_ok);
      ok = ok && c_ok;
      byte |= c << (2 * i);
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// Quantize one warp-held group (4 double-float channels per lane): returns this
// lane's packed byte (channels 4l..4l+3) and the group's fp16 meta.
__device__ __forceinline__ unsigned quantize_warp_df(const DF x[4], float clip, QParams& qp) {
  DF mn, mx;
  warp_minmax_df(x, mn, mx);
  qp = qparams_df(mn, mx, clip);
  return qcode_df(x[0], qp) | (qcode_df(x[1], qp) << 2) | (qcode_df(x[2], qp) << 4) | (qcode_df(x[3], qp) << 6);
}

}  // namespace kvq
