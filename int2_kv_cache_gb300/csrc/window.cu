// Write path of the BF16 sink and recent windows ("Output-Aware Rotation for
// INT2 KV-Cache Quantization", §5 implementation details and Table A; appendix
// "OptR Algorithm" and "Key-mean estimation and application"): the tokens that
// stay in BF16 keep the centred key k - mu (not rotated) and the value
// unchanged; neither is rotated (the decode rotates the window part of its
// readout into the rotated-V basis instead, Eq. 27):
//   key   = bf16_rn(fp32(k - mu))
//   value = bf16_rn(v)          (a copy for bf16 inputs)
// One warp per (window token, KV head); lane l owns channels 4l .. 4l + 3 and
// stores them as 8 bytes of the token's row, at the row's swizzled chunk
// position (chunk c of row r at c ^ r).
#include "kvq_internal.cuh"

namespace kvq {

constexpr int WA_THREADS = 256;

__global__ void __launch_bounds__(WA_THREADS) window_append_kernel(int n_kv_heads, int n_seqs, int max_per_seq,
                                                                   const void* __restrict__ k,
                                                                   const void* __restrict__ v, int dtype,
                                                                   const int32_t* __restrict__ cu_new,
                                                                   const int32_t* __restrict__ start_pos,
                                                                   const float* __restrict__ mu_k, WinGeom win,
                                                                   unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int wi = blockIdx.x * (WA_THREADS / 32) + (threadIdx.x >> 5);
  const int i = wi / n_kv_heads, h = wi % n_kv_heads;
  const int b = blockIdx.y;
  if (i >= max_per_seq || b >= n_seqs) return;
  const int c0 = __ldg(cu_new + b), c1 = __ldg(cu_new + b + 1);
  const int start = __ldg(start_pos + b);
  if (c1 < c0 || start < 0) {
    if (i == 0 && h == 0 && lane == 0) flag_error(err, ERR_SEQ_RANGE);
    return;
  }
  const int end = start + (c1 - c0);
  // new window tokens: the sink part [start, min(S, end)), then the recent part
  // [max(start, S, end - R), end) (disjoint; a slot is written at most once)
  const int n_sink = max(0, min(win.sink, end) - start);
  const int r0 = max(max(start, win.sink), end - win.recent);
  const int n_recent = max(0, end - r0);
  int p;
  if (i < n_sink) p = start + i;
  else if (i - n_sink < n_recent) p = r0 + (i - n_sink);
  else return;
  const int t = c0 + (p - start);
  const int slot = p < win.sink ? p : win.sink + p % win.recent;
  const int n_rec = (win.sink + win.recent) / WIN_REC_TOKENS;
  uint8_t* rec = win.buf + (((size_t)b * n_kv_heads + h) * n_rec + slot / WIN_REC_TOKENS) * WIN_REC_BYTES;
  const int row = slot % WIN_REC_TOKENS;
  const int off = row * 256 + ((((lane >> 1) ^ row)) << 4) + (lane & 1) * 8;
  const size_t elem = ((size_t)t * n_kv_heads + h) * D + 4 * lane;

  // key: one fp32 subtraction, rounded to bf16
  float4 x = load4(k, elem, dtype);
  if (mu_k) {
    const float4 m = __ldg(reinterpret_cast<const float4*>(mu_k + (size_t)h * D) + lane);
    x = make_float4(__fsub_rn(x.x, m.x), __fsub_rn(x.y, m.y), __fsub_rn(x.z, m.z), __fsub_rn(x.w, m.w));
  }
  const __nv_bfloat162 k01 = __floats2bfloat162_rn(x.x, x.y), k23 = __floats2bfloat162_rn(x.z, x.w);
  *reinterpret_cast<uint2*>(rec + off) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&k01), *reinterpret_cast<const uint32_t*>(&k23));

  // value: unchanged, in bf16
  const float4 y = load4(v, elem, dtype);
  const __nv_bfloat162 v01 = __floats2bfloat162_rn(y.x, y.y), v23 = __floats2bfloat162_rn(y.z, y.w);
  *reinterpret_cast<uint2*>(rec + 2048 + off) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&v01), *reinterpret_cast<const uint32_t*>(&v23));
}

cudaError_t launch_window_append(int n_kv_heads, int n_seqs, int n_new, const void* k, const void* v, int dtype,
                                 const int32_t* cu_new, const int32_t* start_pos, const float* mu_k, WinGeom win,
                                 unsigned* err, cudaStream_t s) {
  if (n_new == 0 || n_seqs == 0 || win.sink + win.recent == 0) return cudaSuccess;
  // at most sink + recent window tokens per sequence, and no more than the new tokens
  const int max_per_seq = min(win.sink + win.recent, n_new);
  const long long warps = (long long)max_per_seq * n_kv_heads;
  const dim3 grid((unsigned)((warps + WA_THREADS / 32 - 1) / (WA_THREADS / 32)), n_seqs);
  window_append_kernel<<<grid, WA_THREADS, 0, s>>>(n_kv_heads, n_seqs, max_per_seq, k, v, dtype, cu_new, start_pos,
                                                   mu_k, win, err);
  return cudaGetLastError();
}

}  // namespace kvq
