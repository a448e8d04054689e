// Internal helpers shared by the libkvq translation units (not part of the ABI).
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int D = 128;            // head dimension = quantization group size
constexpr int GROUP_BYTES = 32;   // 128 two-bit codes
constexpr int META_BYTES = 4;     // fp16 scale + fp16 zero

// Device error word bits (read back by kvq_device_check).
enum : unsigned {
  ERR_BLOCK_RANGE = 1u,   // block-table entry outside [0, num_blocks)
  ERR_POS_RANGE = 2u,     // position beyond max_blocks_per_seq * page_tokens
  ERR_SEQ_RANGE = 4u,     // cu_new / seq_lens inconsistent (negative, decreasing, too long)
  ERR_TIMEOUT = 8u,       // a bounded wait on a shared-memory copy gave up
};

struct RotDev {
  int kind;
  const float* signs;
  const float* dense;
};

inline RotDev to_dev(const kvq_rot& r) { return RotDev{r.kind, r.signs, r.dense}; }

// BF16 windows (see kvq_window): sizes in tokens and the record buffer.
struct WinGeom {
  int sink, recent;
  uint8_t* buf;
};
constexpr int WIN_REC_TOKENS = 8;
constexpr int WIN_REC_BYTES = 4096;  // 8 key rows + 8 value rows of 128 bf16

// A decode step's new token (one per sequence, at position seq_lens[b] - 1),
// quantized and written by the decode's query preparation before the decode
// kernel reads the pages (kvq_decode_step).  k, v: [n_seqs][n_kv_heads][128].
struct StepAppend {
  const void* k;
  const void* v;
  int dtype;
  RotDev rot_v;           // the keys use the decode's rot_k
  const float* mu_rot_k;  // mu R_K per head, or nullptr
  float clip_k, clip_v;
  uint8_t* pool;          // the pool, written in place
  WinGeom win;            // BF16 windows (sink + recent = 0: none), written in place
  const float* mu_win;    // the unrotated key mean that centres window keys, or nullptr
};

struct PageGeom {
  int page_tokens;
  int n_kv_heads;
  int num_blocks;
  int max_blocks;
  int record;  // 72 * page_tokens
};

__device__ __forceinline__ void flag_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// Load 4 consecutive channels (16-byte aligned for f32, 8-byte for bf16) as float.
__device__ __forceinline__ float4 load4(const void* base, size_t elem, int dtype) {
  if (dtype == KVQ_F32) {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem));
  }
  uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + elem));
  float4 r;
  r.x = __uint_as_float(w.x << 16);
  r.y = __uint_as_float(w.x & 0xFFFF0000u);
  r.z = __uint_as_float(w.y << 16);
  r.w = __uint_as_float(w.y & 0xFFFF0000u);
  return r;
}

__device__ __forceinline__ float load1(const void* base, size_t elem, int dtype) {
  if (dtype == KVQ_F32) return __ldg(static_cast<const float*>(base) + elem);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[elem]);
}

}  // namespace kvq

// ---- launchers implemented in the kernel translation units (C++ linkage, internal) ----
namespace kvq {

// api.cu: record `msg` as this thread's kvq_last_error() text and return `st`.
kvq_status set_error(kvq_status st, const char* msg);

// api.cu: streaming multiprocessors of the current device (looked up once per
// device ordinal; 152, a GB300's count, if no device can be queried, which only
// sizes workspaces on a machine that cannot launch anyway).
int device_sm_count();

// A kernel's function attributes (its dynamic shared-memory limit) are a
// per-device setting.  `done` keeps one bit per device ordinal below 64; `setup`
// runs on the first call made with a device current (larger ordinals run it on
// every call).  Concurrent first calls may both run it, which is harmless.
template <typename F>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, F&& setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Dynamic shared-memory limit of `kernel`, raised once per device.
template <typename K>
inline cudaError_t smem_limit_once(std::atomic<unsigned long long>& done, K kernel, int bytes) {
  return once_per_device(done, [&] {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
}

// quantize.cu
cudaError_t launch_key_mean(int n_tok, int n_heads, const void* k, int dtype, float* mu,
                            cudaStream_t s);
cudaError_t launch_rotate_heads(int n_rows, int n_heads, int heads_per_rot, const float* x,
                                RotDev rot, float* y, bool transpose, cudaStream_t s);
cudaError_t launch_quantize_append(const PageGeom& g, int n_seqs, int n_new, const void* k,
                                   const void* v, int dtype, const int32_t* cu_new,
                                   const int32_t* start_pos, const int32_t* table, RotDev rot_k,
                                   RotDev rot_v, const float* mu_rot_k, float clip_k, float clip_v,
                                   uint8_t* pool, unsigned* err, cudaStream_t s);
cudaError_t launch_rotate_df(int n_rows, int n_heads, const void* src, int dtype, const float* mu,
                             RotDev rot, float* x_hi, float* x_lo, cudaStream_t s);
cudaError_t launch_quant_dequant(int n_groups, const float* x_hi, const float* x_lo, float clip,
                                 float* out, cudaStream_t s);
// The calibration's private page pool: 16-token pages, records as the decode reads them.
constexpr int CALIB_PAGE = 16;
cudaError_t launch_quant_to_pool(int n_tok, int n_kv_heads, const float* x_hi, const float* x_lo, float clip,
                                 int role, uint8_t* pool, cudaStream_t s);

// window.cu
cudaError_t launch_window_append(int n_kv_heads, int n_seqs, int n_new, const void* k, const void* v,
                                 int dtype, const int32_t* cu_new, const int32_t* start_pos,
                                 const float* mu_k, WinGeom win, unsigned* err, cudaStream_t s);

// decode.cu (win.sink = win.recent = 0: no windows)
int decode_auto_ctas(int n_seqs, int n_kv_heads, int gqa, int max_seq_len);
size_t decode_workspace_bytes(int n_seqs, int n_kv_heads, int gqa, int n_ctas, bool windows = false);
cudaError_t launch_decode(const PageGeom& g, int n_q_heads, int n_seqs, const void* q,
                          int q_dtype, const int32_t* seq_lens, int max_seq_len,
                          const int32_t* table, RotDev rot_k, const uint8_t* pool, int n_ctas,
                          void* ws, float* o_rot, unsigned* err, cudaStream_t s,
                          WinGeom win = WinGeom{0, 0, nullptr}, RotDev rot_v = RotDev{0, nullptr, nullptr},
                          const StepAppend* app = nullptr);

// outproj.cu
cudaError_t launch_fold_wo(int d_model, int n_q_heads, int gqa, const void* w, int w_dtype,
                           RotDev rot_v, void* out, int out_dtype, cudaStream_t s);
cudaError_t launch_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                            int w_dtype, float* y, unsigned* err, cudaStream_t s);
size_t wo_packed_bytes(int d_model, int k_dim);
cudaError_t launch_pack_wo(int d_model, int k_dim, const void* w, void* out, cudaStream_t s);
cudaError_t launch_out_proj_packed(int n_rows, int d_model, int k_dim, const float* x, const void* w_packed, float* y,
                                   unsigned* err, cudaStream_t s);

// optr.cu: OptR calibration of one KV head (fp64)
struct OptrTraceIn {  // one trace of the head: q [n_qpos][gqa][128], k, v [n_tok][128] (fp32)
  const float* q;
  const float* k;
  const float* v;
  int n_tok, n_qpos;
};
size_t optr_workspace_bytes(int n_tok, int n_qpos, int n_tok_h, int n_qpos_h, int gqa);
cudaError_t launch_optr_loss_grad(int phase, const OptrTraceIn& tr, int gqa, int d_model, const float* w_o,
                                  const float* mu, const double* r0, const double* a, const double* r_k_sel,
                                  float clip_k, float clip_v, float lam, double* loss, double* grad, void* ws,
                                  unsigned* err, cudaStream_t s);
cudaError_t launch_optr_calibrate(const OptrTraceIn& tr, const OptrTraceIn* ho, int gqa, int d_model,
                                  const float* w_o, const float* mu, const double* r_k0, const double* r_v0,
                                  float clip_k, float clip_v, float lam, int steps, float lr, int every, double* r_k,
                                  double* r_v, double* loss_k, double* loss_v, void* ws, unsigned* err,
                                  cudaStream_t s);

// calib.cu
size_t calib_workspace_bytes(int n_tok, int n_qpos, int n_kv_heads, int gqa, int joint);
size_t report_workspace_bytes(int n_tok, int n_qpos, int n_kv_heads, int gqa);
cudaError_t launch_head_report(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model, const void* q,
                               const void* k, const void* v, int dtype, const void* w_o, int w_dtype, RotDev rot_k,
                               RotDev rot_v, const float* mu, float clip_k, float clip_v, double* out, void* ws,
                               unsigned* err, cudaStream_t s);
cudaError_t launch_calib(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model,
                         const void* q, const void* k, const void* v, int dtype, const void* w_o,
                         int w_dtype, int n_cand, const kvq_rot* cand, int n_clip,
                         const float* clips, const float* mu, int joint, double* nmse,
                         double* ref, void* ws, unsigned* err, cudaStream_t s);

}  // namespace kvq
