// Group quantizer shared by the write path and the calibration sweep.
//
// One group = the 128 channels of one token of one head ("Output-Aware Rotation
// for INT2 KV-Cache Quantization", §3.1 Eq. 4 and §5 implementation details:
// group-wise affine INT2, group size 128, clip ratio c; fp16 scale and zero as
// the 2.32 bits-per-element accounting implies):
//   lo = c * min(x), hi = c * max(x)
//   scale = fp16_rn((hi - lo) / 3), zero = fp16_rn(lo)
//   code  = clamp(rint((x - zero) / scale), 0, 3), 0 where scale == 0
// Arithmetic is fp32; (x - zero) / scale is evaluated as (x - zero) * (1 / scale)
// with an IEEE reciprocal (at most ~2 ulp from the quotient).
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

struct QParams {
  unsigned short s_bits, z_bits;
  float s, z, r;  // fp16-rounded scale and zero (as float), reciprocal of s (0 if s == 0)
};

__device__ __forceinline__ QParams qparams(float mn, float mx, float clip) {
  float lo = clip * mn;
  float hi = clip * mx;
  float sc = __fdiv_rn(hi - lo, 3.0f);
  __half s16 = __float2half_rn(sc);
  __half z16 = __float2half_rn(lo);
  QParams p;
  p.s_bits = __half_as_ushort(s16);
  p.z_bits = __half_as_ushort(z16);
  p.s = __half2float(s16);
  p.z = __half2float(z16);
  p.r = p.s > 0.f ? __frcp_rn(p.s) : 0.f;
  return p;
}

__device__ __forceinline__ unsigned qcode(float x, const QParams& p) {
  int c = __float2int_rn((x - p.z) * p.r);
  c = c < 0 ? 0 : (c > 3 ? 3 : c);
  return p.s > 0.f ? (unsigned)c : 0u;
}

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

// Warp-cooperative Walsh-Hadamard transform of 128 values, lane l holding
// channels 4l..4l+3 (Sylvester order, unnormalised): two butterfly stages in
// registers, five across lanes.
__device__ __forceinline__ void warp_fwht128(float4& v, int lane) {
  float a0 = v.x + v.y, a1 = v.x - v.y, a2 = v.z + v.w, a3 = v.z - v.w;
  v.x = a0 + a2; v.z = a0 - a2; v.y = a1 + a3; v.w = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    float px = __shfl_xor_sync(0xffffffffu, v.x, m);
    float py = __shfl_xor_sync(0xffffffffu, v.y, m);
    float pz = __shfl_xor_sync(0xffffffffu, v.z, m);
    float pw = __shfl_xor_sync(0xffffffffu, v.w, m);
    if (lane & m) { v.x = px - v.x; v.y = py - v.y; v.z = pz - v.z; v.w = pw - v.w; }
    else          { v.x = v.x + px; v.y = v.y + py; v.z = v.z + pz; v.w = v.w + pw; }
  }
}

// 1 / sqrt(128) rounded to fp32.
constexpr float INV_SQRT_D = 0.08838834764831845f;

// Rotate one head vector held by a warp (lane l owns channels 4l..4l+3):
// y = x R_head, or y = x R_head^T when `transpose`.
__device__ __forceinline__ float4 rotate_vec_warp(float4 v, const RotDev& rot, int head, int lane,
                                                  bool transpose) {
  if (rot.kind == KVQ_ROT_SIGNED_HADAMARD) {
    const float4 s = __ldg(reinterpret_cast<const float4*>(rot.signs + (size_t)head * D) + lane);
    if (!transpose) { v.x *= s.x; v.y *= s.y; v.z *= s.z; v.w *= s.w; }
    warp_fwht128(v, lane);
    v.x *= INV_SQRT_D; v.y *= INV_SQRT_D; v.z *= INV_SQRT_D; v.w *= INV_SQRT_D;
    if (transpose) { v.x *= s.x; v.y *= s.y; v.z *= s.z; v.w *= s.w; }
    return v;
  }
  if (rot.kind == KVQ_ROT_DENSE) {
    const float* R = rot.dense + (size_t)head * D * D;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!transpose) {
      // y_d = sum_c x_c R[c][d], lane owns d = 4*lane .. 4*lane+3
#pragma unroll 4
      for (int c = 0; c < D; ++c) {
        float src = (c & 3) == 0 ? v.x : (c & 3) == 1 ? v.y : (c & 3) == 2 ? v.z : v.w;
        float xc = __shfl_sync(0xffffffffu, src, c >> 2);
        float4 r = __ldg(reinterpret_cast<const float4*>(R + (size_t)c * D) + lane);
        y.x = fmaf(xc, r.x, y.x); y.y = fmaf(xc, r.y, y.y);
        y.z = fmaf(xc, r.z, y.z); y.w = fmaf(xc, r.w, y.w);
      }
    } else {
      // y_d = sum_c x_c R[d][c]
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4* row = reinterpret_cast<const float4*>(R + (size_t)(4 * lane + i) * D);
        float part = 0.f;
        for (int c4 = 0; c4 < 32; ++c4) {
          float4 r = __ldg(row + c4);
          float x0 = __shfl_sync(0xffffffffu, v.x, c4), x1 = __shfl_sync(0xffffffffu, v.y, c4);
          float x2 = __shfl_sync(0xffffffffu, v.z, c4), x3 = __shfl_sync(0xffffffffu, v.w, c4);
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


}  // namespace kvq
