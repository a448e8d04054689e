// libkvq C ABI: argument validation, typed status codes, the device error word,
// and dispatch to the kernel launchers.  See include/kvq.h for the contract of
// every entry point.
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <mutex>
#include <string>

#include "kvq_internal.cuh"

namespace {

thread_local std::string g_last_error = "no error";

kvq_status fail(kvq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kvq_status cuda_fail(cudaError_t e, const char* where) {
  return fail(KVQ_ECUDA, "%s: CUDA error %d (%s)", where, (int)e, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int dt) { return dt == KVQ_F32 || dt == KVQ_BF16; }

bool valid_clip(float c) { return std::isfinite(c) && c > 0.f && c <= 1.f; }

}  // namespace

// One error word per device; its address is looked up once per device.
__device__ unsigned kvq_device_error_word;

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_err_mutex;
unsigned* g_err_addr[MAX_DEVICES] = {nullptr};

kvq_status device_error_word(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= MAX_DEVICES) return fail(KVQ_EUNSUPPORTED, "device ordinal %d >= %d", dev, MAX_DEVICES);
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (!g_err_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, kvq_device_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    g_err_addr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_addr[dev];
  return KVQ_OK;
}

kvq_status check_layout(const kvq_layout* L, bool decode) {
  if (!L) return fail(KVQ_EINVAL, "layout is NULL");
  if (L->head_dim != kvq::D) return fail(KVQ_EUNSUPPORTED, "head_dim %d: only 128 is supported", L->head_dim);
  if (L->page_tokens != 8 && L->page_tokens != 16)
    return fail(KVQ_EUNSUPPORTED, "page_tokens %d: only 8 or 16 are supported", L->page_tokens);
  if (L->n_kv_heads < 1) return fail(KVQ_EINVAL, "n_kv_heads %d < 1", L->n_kv_heads);
  if (L->n_q_heads < 1 || L->n_q_heads % L->n_kv_heads != 0)
    return fail(KVQ_EINVAL, "n_q_heads %d is not a positive multiple of n_kv_heads %d", L->n_q_heads, L->n_kv_heads);
  if (decode) {
    const int g = L->n_q_heads / L->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8)
      return fail(KVQ_EUNSUPPORTED, "query heads per KV head %d: supported 1, 2, 4, 8", g);
  }
  if (L->num_blocks < 1) return fail(KVQ_EINVAL, "num_blocks %d < 1", L->num_blocks);
  if (L->max_blocks_per_seq < 1) return fail(KVQ_EINVAL, "max_blocks_per_seq %d < 1", L->max_blocks_per_seq);
  return KVQ_OK;
}

kvq_status check_rot(const kvq_rot& r, const char* name) {
  switch (r.kind) {
    case KVQ_ROT_IDENTITY: return KVQ_OK;
    case KVQ_ROT_SIGNED_HADAMARD:
      if (!r.signs || !aligned16(r.signs)) return fail(KVQ_EINVAL, "%s: signs NULL or not 16-byte aligned", name);
      return KVQ_OK;
    case KVQ_ROT_DENSE:
      if (!r.dense || !aligned16(r.dense)) return fail(KVQ_EINVAL, "%s: dense NULL or not 16-byte aligned", name);
      return KVQ_OK;
    default: return fail(KVQ_EINVAL, "%s: unknown rotation kind %d", name, r.kind);
  }
}

// Window sizes (kvq_window); *out = no windows for NULL or two zero sizes.
kvq_status check_window(const kvq_window* w, kvq::WinGeom* out) {
  *out = kvq::WinGeom{0, 0, nullptr};
  if (!w || (w->sink_tokens == 0 && w->recent_tokens == 0)) return KVQ_OK;
  if (w->sink_tokens < 0 || w->sink_tokens % 64 != 0)
    return fail(KVQ_EINVAL, "window sink_tokens %d is not a non-negative multiple of 64", w->sink_tokens);
  if (w->recent_tokens < 0 || w->recent_tokens % 8 != 0)
    return fail(KVQ_EINVAL, "window recent_tokens %d is not a non-negative multiple of 8", w->recent_tokens);
  if (w->sink_tokens + w->recent_tokens > 65536)
    return fail(KVQ_EUNSUPPORTED, "window of %d tokens > 65536", w->sink_tokens + w->recent_tokens);
  if (!w->buf || !aligned16(w->buf)) return fail(KVQ_EINVAL, "window buf is NULL or not 16-byte aligned");
  *out = kvq::WinGeom{w->sink_tokens, w->recent_tokens, w->buf};
  return KVQ_OK;
}

kvq::PageGeom geom(const kvq_layout* L) {
  return kvq::PageGeom{L->page_tokens, L->n_kv_heads, L->num_blocks, L->max_blocks_per_seq,
                       72 * L->page_tokens};
}

#define KVQ_CHECK(expr)             \
  do {                              \
    kvq_status st_ = (expr);        \
    if (st_ != KVQ_OK) return st_;  \
  } while (0)

#define KVQ_IDX(p, name)                                                               \
  do {                                                                                 \
    if (!(p)) return fail(KVQ_EINVAL, "%s is NULL", name);                             \
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0)                                    \
      return fail(KVQ_EINVAL, "%s is not 4-byte aligned", name);                       \
  } while (0)

#define KVQ_PTR(p, name)                                                         \
  do {                                                                           \
    if (!(p)) return fail(KVQ_EINVAL, "%s is NULL", name);                       \
    if (!aligned16(p)) return fail(KVQ_EINVAL, "%s is not 16-byte aligned", name); \
  } while (0)

}  // namespace

kvq_status kvq::set_error(kvq_status st, const char* msg) { return fail(st, "%s", msg); }

int kvq::device_sm_count() {
  static std::atomic<int> cache[64];  // per device ordinal, 0 = not yet looked up
  int dev = 0, c = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();  // leave no error behind for the caller's launch checks
    return 152;
  }
  if (dev >= 0 && dev < 64 && (c = cache[dev].load(std::memory_order_relaxed)) > 0) return c;
  if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(c, std::memory_order_relaxed);
  return c;
}

extern "C" {

const char* kvq_last_error(void) { return g_last_error.c_str(); }

size_t kvq_pool_bytes(const kvq_layout* L) {
  if (!L || L->num_blocks < 0 || L->n_kv_heads < 0 || L->page_tokens < 0) return 0;
  return (size_t)L->num_blocks * L->n_kv_heads * 72 * L->page_tokens;
}

kvq_status kvq_device_check(kvq_stream stream) {
  unsigned* addr = nullptr;
  KVQ_CHECK(device_error_word(&addr));
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, addr, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (word == 0) return KVQ_OK;
  const unsigned zero = 0;
  e = cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  return fail(KVQ_EDEVICE_FLAG, "kernel bounds check fired (0x%x):%s%s%s", word,
              (word & kvq::ERR_BLOCK_RANGE) ? " block-table entry out of range;" : "",
              (word & kvq::ERR_POS_RANGE) ? " position beyond the block table;" : "",
              (word & kvq::ERR_SEQ_RANGE) ? " inconsistent cu_new/seq_lens;" : "");
}

kvq_status kvq_key_mean(int n_tok, int n_kv_heads, const void* k, kvq_dtype dtype, float* mu,
                        kvq_stream stream) {
  if (n_tok < 1 || n_kv_heads < 1) return fail(KVQ_EINVAL, "n_tok %d / n_kv_heads %d must be >= 1", n_tok, n_kv_heads);
  if (!valid_dtype(dtype)) return fail(KVQ_EINVAL, "bad dtype %d", (int)dtype);
  KVQ_PTR(k, "k");
  KVQ_PTR(mu, "mu");
  cudaError_t e = kvq::launch_key_mean(n_tok, n_kv_heads, k, dtype, mu, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_key_mean");
}

kvq_status kvq_rotate_heads(int n_rows, int n_heads, int heads_per_rot, const float* x, kvq_rot rot,
                            float* y, kvq_stream stream) {
  if (n_rows < 0 || n_heads < 1 || heads_per_rot < 1 || n_heads % heads_per_rot != 0)
    return fail(KVQ_EINVAL, "bad shape n_rows %d n_heads %d heads_per_rot %d", n_rows, n_heads, heads_per_rot);
  KVQ_CHECK(check_rot(rot, "rot"));
  if (n_rows == 0) return KVQ_OK;
  KVQ_PTR(x, "x");
  KVQ_PTR(y, "y");
  if (x == y) return fail(KVQ_EINVAL, "x and y must not alias");
  cudaError_t e = kvq::launch_rotate_heads(n_rows, n_heads, heads_per_rot, x, kvq::to_dev(rot), y, false, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_rotate_heads");
}

kvq_status kvq_quantize_append(const kvq_layout* layout, int n_seqs, int n_new_total, const void* k,
                               const void* v, kvq_dtype dtype, const int32_t* cu_new,
                               const int32_t* start_pos, const int32_t* block_table, kvq_rot rot_k,
                               kvq_rot rot_v, const float* mu_rot_k, float clip_k, float clip_v,
                               uint8_t* pool, kvq_stream stream) {
  KVQ_CHECK(check_layout(layout, false));
  if (n_seqs < 1) return fail(KVQ_EINVAL, "n_seqs %d < 1", n_seqs);
  if (n_new_total < 0) return fail(KVQ_EINVAL, "n_new_total %d < 0", n_new_total);
  if (!valid_dtype(dtype)) return fail(KVQ_EINVAL, "bad dtype %d", (int)dtype);
  if (!valid_clip(clip_k) || !valid_clip(clip_v))
    return fail(KVQ_EINVAL, "clip ratios must lie in (0, 1] (got %g, %g)", clip_k, clip_v);
  KVQ_CHECK(check_rot(rot_k, "rot_k"));
  KVQ_CHECK(check_rot(rot_v, "rot_v"));
  if (n_new_total == 0) return KVQ_OK;
  KVQ_PTR(k, "k");
  KVQ_PTR(v, "v");
  KVQ_IDX(cu_new, "cu_new");
  KVQ_IDX(start_pos, "start_pos");
  KVQ_IDX(block_table, "block_table");
  KVQ_PTR(pool, "pool");
  if (mu_rot_k && !aligned16(mu_rot_k)) return fail(KVQ_EINVAL, "mu_rot_k is not 16-byte aligned");
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  const kvq::PageGeom g = geom(layout);
  cudaError_t e = kvq::launch_quantize_append(g, n_seqs, n_new_total, k, v, dtype, cu_new, start_pos,
                                              block_table, kvq::to_dev(rot_k), kvq::to_dev(rot_v), mu_rot_k,
                                              clip_k, clip_v, pool, err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_quantize_append");
}

kvq_status kvq_window_append(const kvq_layout* layout, int n_seqs, int n_new_total, const void* k,
                             const void* v, kvq_dtype dtype, const int32_t* cu_new, const int32_t* start_pos,
                             const float* mu_k, const kvq_window* win, kvq_stream stream) {
  KVQ_CHECK(check_layout(layout, false));
  if (n_seqs < 1 || n_seqs > 65535) return fail(KVQ_EINVAL, "n_seqs %d outside [1, 65535]", n_seqs);
  if (n_new_total < 0) return fail(KVQ_EINVAL, "n_new_total %d < 0", n_new_total);
  if (!valid_dtype(dtype)) return fail(KVQ_EINVAL, "bad dtype %d", (int)dtype);
  kvq::WinGeom wg;
  KVQ_CHECK(check_window(win, &wg));
  if (n_new_total == 0 || wg.sink + wg.recent == 0) return KVQ_OK;
  KVQ_PTR(k, "k");
  KVQ_PTR(v, "v");
  KVQ_IDX(cu_new, "cu_new");
  KVQ_IDX(start_pos, "start_pos");
  if (mu_k && !aligned16(mu_k)) return fail(KVQ_EINVAL, "mu_k is not 16-byte aligned");
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  cudaError_t e = kvq::launch_window_append(layout->n_kv_heads, n_seqs, n_new_total, k, v, dtype, cu_new, start_pos,
                                            mu_k, wg, err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_window_append");
}

// Index ranges the decode kernels keep in 32-bit integers.
static kvq_status check_decode_size(const kvq_layout* layout, int n_seqs, int max_seq_len) {
  if (n_seqs > 65535) return fail(KVQ_EUNSUPPORTED, "n_seqs %d > 65535", n_seqs);
  const long long entries = (long long)n_seqs * layout->n_kv_heads * ((max_seq_len + 31) / 32);
  if (entries >= (1ll << 30)) return fail(KVQ_EUNSUPPORTED, "%lld cached 32-token chunks per call", entries);
  if ((long long)layout->num_blocks * layout->n_kv_heads >= (1ll << 31))
    return fail(KVQ_EUNSUPPORTED, "num_blocks * n_kv_heads >= 2^31");
  if ((long long)layout->max_blocks_per_seq * layout->page_tokens >= (1ll << 31))
    return fail(KVQ_EUNSUPPORTED, "max_blocks_per_seq * page_tokens >= 2^31");
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_size(const kvq_layout* layout, int n_seqs, int max_seq_len,
                                     int n_splits, size_t* bytes) {
  return kvq_decode_workspace_size_win(layout, n_seqs, max_seq_len, n_splits, nullptr, bytes);
}

kvq_status kvq_decode_workspace_size_win(const kvq_layout* layout, int n_seqs, int max_seq_len, int n_splits,
                                         const kvq_window* win, size_t* bytes) {
  KVQ_CHECK(check_layout(layout, true));
  kvq::WinGeom wg;
  KVQ_CHECK(check_window(win, &wg));
  if (!bytes) return fail(KVQ_EINVAL, "bytes is NULL");
  if (n_seqs < 0 || max_seq_len < 0 || n_splits < 0 || n_splits > 8192)
    return fail(KVQ_EINVAL, "bad n_seqs %d / max_seq_len %d / n_splits %d", n_seqs, max_seq_len, n_splits);
  KVQ_CHECK(check_decode_size(layout, n_seqs, max_seq_len));
  const int gqa = layout->n_q_heads / layout->n_kv_heads;
  const int s = n_splits ? n_splits : kvq::decode_auto_ctas(n_seqs, layout->n_kv_heads, gqa, max_seq_len);
  *bytes = kvq::decode_workspace_bytes(n_seqs, layout->n_kv_heads, gqa, s, wg.sink + wg.recent > 0);
  return KVQ_OK;
}

kvq_status kvq_decode_attention(const kvq_layout* layout, int n_seqs, const void* q, kvq_dtype q_dtype,
                                const int32_t* seq_lens, int max_seq_len, const int32_t* block_table,
                                kvq_rot rot_k, const uint8_t* pool, int n_splits, void* workspace,
                                size_t workspace_bytes, float* o_rot, kvq_stream stream) {
  const kvq_rot identity = {KVQ_ROT_IDENTITY, nullptr, nullptr};
  return kvq_decode_attention_win(layout, n_seqs, q, q_dtype, seq_lens, max_seq_len, block_table, rot_k, identity,
                                  pool, nullptr, n_splits, workspace, workspace_bytes, o_rot, stream);
}

}  // extern "C"

static kvq_status decode_step_impl(const char* name, const kvq_layout* layout, int n_seqs, const void* q,
                                   const void* k_new, const void* v_new, kvq_dtype dtype, const int32_t* seq_lens,
                                   int max_seq_len, const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v,
                                   const float* mu_rot_k, float clip_k, float clip_v, uint8_t* pool,
                                   const kvq_window* win, const float* mu_k, int n_splits, void* workspace,
                                   size_t workspace_bytes, float* o_rot, kvq_stream stream) {
  KVQ_CHECK(check_layout(layout, true));
  kvq::WinGeom wg;
  KVQ_CHECK(check_window(win, &wg));
  const bool windows = wg.sink + wg.recent > 0;
  if (n_seqs < 0) return fail(KVQ_EINVAL, "n_seqs %d < 0", n_seqs);
  if (!valid_dtype(dtype)) return fail(KVQ_EINVAL, "bad dtype %d", (int)dtype);
  if (!valid_clip(clip_k) || !valid_clip(clip_v))
    return fail(KVQ_EINVAL, "clip ratios must lie in (0, 1] (got %g, %g)", clip_k, clip_v);
  if (max_seq_len < 0 || (long long)max_seq_len > (long long)layout->max_blocks_per_seq * layout->page_tokens)
    return fail(KVQ_EINVAL, "max_seq_len %d outside [0, max_blocks_per_seq * page_tokens]", max_seq_len);
  if (n_splits < 0 || n_splits > 8192) return fail(KVQ_EINVAL, "n_splits %d outside [0, 8192]", n_splits);
  KVQ_CHECK(check_rot(rot_k, "rot_k"));
  KVQ_CHECK(check_rot(rot_v, "rot_v"));
  if (n_seqs == 0) return KVQ_OK;
  KVQ_PTR(q, "q");
  KVQ_PTR(k_new, "k_new");
  KVQ_PTR(v_new, "v_new");
  KVQ_IDX(seq_lens, "seq_lens");
  KVQ_IDX(block_table, "block_table");
  KVQ_PTR(pool, "pool");
  KVQ_PTR(o_rot, "o_rot");
  KVQ_PTR(workspace, "workspace");
  if (mu_rot_k && !aligned16(mu_rot_k)) return fail(KVQ_EINVAL, "mu_rot_k is not 16-byte aligned");
  if (mu_k && !aligned16(mu_k)) return fail(KVQ_EINVAL, "mu_k is not 16-byte aligned");
  KVQ_CHECK(check_decode_size(layout, n_seqs, max_seq_len));
  const int gqa = layout->n_q_heads / layout->n_kv_heads;
  const int s = n_splits ? n_splits : kvq::decode_auto_ctas(n_seqs, layout->n_kv_heads, gqa, max_seq_len);
  const size_t need = kvq::decode_workspace_bytes(n_seqs, layout->n_kv_heads, gqa, s, windows);
  if (workspace_bytes < need)
    return fail(KVQ_EINVAL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  const kvq::StepAppend app{k_new, v_new, (int)dtype, kvq::to_dev(rot_v), mu_rot_k, clip_k, clip_v, pool, wg, mu_k};
  cudaError_t e = kvq::launch_decode(geom(layout), layout->n_q_heads, n_seqs, q, dtype, seq_lens, max_seq_len,
                                     block_table, kvq::to_dev(rot_k), pool, s, workspace, o_rot, err, stream, wg,
                                     kvq::to_dev(rot_v), &app);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, name);
}

extern "C" {

kvq_status kvq_decode_step(const kvq_layout* layout, int n_seqs, const void* q, const void* k_new,
                           const void* v_new, kvq_dtype dtype, const int32_t* seq_lens, int max_seq_len,
                           const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v, const float* mu_rot_k,
                           float clip_k, float clip_v, uint8_t* pool, int n_splits, void* workspace,
                           size_t workspace_bytes, float* o_rot, kvq_stream stream) {
  return decode_step_impl("kvq_decode_step", layout, n_seqs, q, k_new, v_new, dtype, seq_lens, max_seq_len,
                          block_table, rot_k, rot_v, mu_rot_k, clip_k, clip_v, pool, nullptr, nullptr, n_splits,
                          workspace, workspace_bytes, o_rot, stream);
}

kvq_status kvq_decode_step_win(const kvq_layout* layout, int n_seqs, const void* q, const void* k_new,
                               const void* v_new, kvq_dtype dtype, const int32_t* seq_lens, int max_seq_len,
                               const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v, const float* mu_rot_k,
                               const float* mu_k, float clip_k, float clip_v, uint8_t* pool, const kvq_window* win,
                               int n_splits, void* workspace, size_t workspace_bytes, float* o_rot,
                               kvq_stream stream) {
  return decode_step_impl("kvq_decode_step_win", layout, n_seqs, q, k_new, v_new, dtype, seq_lens, max_seq_len,
                          block_table, rot_k, rot_v, mu_rot_k, clip_k, clip_v, pool, win, mu_k, n_splits, workspace,
                          workspace_bytes, o_rot, stream);
}

static kvq_status check_optr_trace(const kvq_optr_trace* t, const char* name, int gqa) {
  if (!t) return fail(KVQ_EINVAL, "%s is NULL", name);
  if (t->n_tok < 1 || t->n_tok > 8192) return fail(KVQ_EUNSUPPORTED, "%s: n_tok %d outside [1, 8192]", name, t->n_tok);
  if (t->n_qpos < 1 || t->n_qpos > t->n_tok)
    return fail(KVQ_EINVAL, "%s: n_qpos %d outside [1, n_tok]", name, t->n_qpos);
  if ((long long)t->n_qpos * gqa > 65535) return fail(KVQ_EUNSUPPORTED, "%s: n_qpos * gqa > 65535", name);
  KVQ_PTR(t->q, "trace q");
  KVQ_PTR(t->k, "trace k");
  KVQ_PTR(t->v, "trace v");
  return KVQ_OK;
}

static kvq_status check_optr_common(int gqa, int d_model, const float* w_o, const float* mu) {
  if (gqa < 1 || gqa > 64) return fail(KVQ_EINVAL, "gqa %d outside [1, 64]", gqa);
  if (d_model < 1 || d_model > 8192) return fail(KVQ_EUNSUPPORTED, "d_model %d outside [1, 8192]", d_model);
  KVQ_PTR(w_o, "w_o");
  if (mu && !aligned16(mu)) return fail(KVQ_EINVAL, "mu is not 16-byte aligned");
  return KVQ_OK;
}

kvq_status kvq_optr_workspace_size(int n_tok, int n_qpos, int n_tok_heldout, int n_qpos_heldout, int gqa,
                                   size_t* bytes) {
  if (!bytes) return fail(KVQ_EINVAL, "bytes is NULL");
  if (n_tok < 1 || n_qpos < 1 || gqa < 1 || n_tok_heldout < 0 || n_qpos_heldout < 0)
    return fail(KVQ_EINVAL, "bad sizes");
  *bytes = kvq::optr_workspace_bytes(n_tok, n_qpos, n_tok_heldout, n_qpos_heldout, gqa);
  return KVQ_OK;
}

kvq_status kvq_optr_loss_grad(int phase, const kvq_optr_trace* trace, int gqa, int d_model, const float* w_o,
                              const float* mu, const double* r0, const double* a, const double* r_k_sel,
                              float clip_k, float clip_v, float lambda_k, double* loss, double* grad,
                              void* workspace, size_t workspace_bytes, kvq_stream stream) {
  if (phase != KVQ_OPTR_KEYS && phase != KVQ_OPTR_VALUES) return fail(KVQ_EINVAL, "phase %d", phase);
  KVQ_CHECK(check_optr_trace(trace, "trace", gqa));
  KVQ_CHECK(check_optr_common(gqa, d_model, w_o, mu));
  if (!valid_clip(clip_k) || !valid_clip(clip_v))
    return fail(KVQ_EINVAL, "clip ratios must lie in (0, 1] (got %g, %g)", clip_k, clip_v);
  if (!std::isfinite(lambda_k)) return fail(KVQ_EINVAL, "lambda_k is not finite");
  KVQ_PTR(r0, "r0");
  KVQ_PTR(a, "a");
  if (phase == KVQ_OPTR_VALUES) KVQ_PTR(r_k_sel, "r_k_sel");
  if (!loss || (reinterpret_cast<uintptr_t>(loss) & 7u)) return fail(KVQ_EINVAL, "loss is NULL or not 8-byte aligned");
  if (grad && !aligned16(grad)) return fail(KVQ_EINVAL, "grad is not 16-byte aligned");
  KVQ_PTR(workspace, "workspace");
  const size_t need = kvq::optr_workspace_bytes(trace->n_tok, trace->n_qpos, 0, 0, gqa);
  if (workspace_bytes < need) return fail(KVQ_EINVAL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  const kvq::OptrTraceIn tr{trace->q, trace->k, trace->v, trace->n_tok, trace->n_qpos};
  cudaError_t e = kvq::launch_optr_loss_grad(phase, tr, gqa, d_model, w_o, mu, r0, a, r_k_sel, clip_k, clip_v,
                                             lambda_k, loss, grad, workspace, err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_optr_loss_grad");
}

kvq_status kvq_optr_calibrate_head(const kvq_optr_trace* train, const kvq_optr_trace* heldout, int gqa, int d_model,
                                   const float* w_o, const float* mu, const double* r_k0, const double* r_v0,
                                   float clip_k, float clip_v, float lambda_k, int steps, float lr, int every,
                                   double* r_k, double* r_v, double* loss_k, double* loss_v, void* workspace,
                                   size_t workspace_bytes, kvq_stream stream) {
  KVQ_CHECK(check_optr_trace(train, "train", gqa));
  if (heldout) KVQ_CHECK(check_optr_trace(heldout, "heldout", gqa));
  KVQ_CHECK(check_optr_common(gqa, d_model, w_o, mu));
  if (!valid_clip(clip_k) || !valid_clip(clip_v))
    return fail(KVQ_EINVAL, "clip ratios must lie in (0, 1] (got %g, %g)", clip_k, clip_v);
  if (!std::isfinite(lambda_k) || !std::isfinite(lr) || !(lr > 0.f)) return fail(KVQ_EINVAL, "bad lambda_k or lr");
  if (steps < 0 || steps > 100000 || every < 0) return fail(KVQ_EINVAL, "bad steps %d / every %d", steps, every);
  KVQ_PTR(r_k0, "r_k0");
  KVQ_PTR(r_v0, "r_v0");
  KVQ_PTR(r_k, "r_k");
  KVQ_PTR(r_v, "r_v");
  if (loss_k && (reinterpret_cast<uintptr_t>(loss_k) & 7u)) return fail(KVQ_EINVAL, "loss_k not 8-byte aligned");
  if (loss_v && (reinterpret_cast<uintptr_t>(loss_v) & 7u)) return fail(KVQ_EINVAL, "loss_v not 8-byte aligned");
  KVQ_PTR(workspace, "workspace");
  const size_t need = kvq::optr_workspace_bytes(train->n_tok, train->n_qpos, heldout ? heldout->n_tok : 0,
                                                heldout ? heldout->n_qpos : 0, gqa);
  if (workspace_bytes < need) return fail(KVQ_EINVAL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  const kvq::OptrTraceIn tr{train->q, train->k, train->v, train->n_tok, train->n_qpos};
  kvq::OptrTraceIn ho{};
  if (heldout) ho = kvq::OptrTraceIn{heldout->q, heldout->k, heldout->v, heldout->n_tok, heldout->n_qpos};
  cudaError_t e = kvq::launch_optr_calibrate(tr, heldout ? &ho : nullptr, gqa, d_model, w_o, mu, r_k0, r_v0, clip_k,
                                             clip_v, lambda_k, steps, lr, every, r_k, r_v, loss_k, loss_v, workspace,
                                             err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_optr_calibrate_head");
}

kvq_status kvq_decode_attention_win(const kvq_layout* layout, int n_seqs, const void* q, kvq_dtype q_dtype,
                                    const int32_t* seq_lens, int max_seq_len, const int32_t* block_table,
                                    kvq_rot rot_k, kvq_rot rot_v, const uint8_t* pool, const kvq_window* win,
                                    int n_splits, void* workspace, size_t workspace_bytes, float* o_rot,
                                    kvq_stream stream) {
  KVQ_CHECK(check_layout(layout, true));
  kvq::WinGeom wg;
  KVQ_CHECK(check_window(win, &wg));
  KVQ_CHECK(check_rot(rot_v, "rot_v"));
  if (n_seqs < 0) return fail(KVQ_EINVAL, "n_seqs %d < 0", n_seqs);
  if (!valid_dtype(q_dtype)) return fail(KVQ_EINVAL, "bad q dtype %d", (int)q_dtype);
  if (max_seq_len < 0 || (long long)max_seq_len > (long long)layout->max_blocks_per_seq * layout->page_tokens)
    return fail(KVQ_EINVAL, "max_seq_len %d outside [0, max_blocks_per_seq * page_tokens]", max_seq_len);
  if (n_splits < 0 || n_splits > 8192) return fail(KVQ_EINVAL, "n_splits %d outside [0, 8192]", n_splits);
  KVQ_CHECK(check_rot(rot_k, "rot_k"));
  if (n_seqs == 0) return KVQ_OK;
  KVQ_PTR(q, "q");
  KVQ_IDX(seq_lens, "seq_lens");
  KVQ_IDX(block_table, "block_table");
  KVQ_PTR(pool, "pool");
  KVQ_PTR(o_rot, "o_rot");
  KVQ_PTR(workspace, "workspace");
  KVQ_CHECK(check_decode_size(layout, n_seqs, max_seq_len));
  const int gqa = layout->n_q_heads / layout->n_kv_heads;
  const int s = n_splits ? n_splits : kvq::decode_auto_ctas(n_seqs, layout->n_kv_heads, gqa, max_seq_len);
  const size_t need = kvq::decode_workspace_bytes(n_seqs, layout->n_kv_heads, gqa, s, wg.sink + wg.recent > 0);
  if (workspace_bytes < need)
    return fail(KVQ_EINVAL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  cudaError_t e = kvq::launch_decode(geom(layout), layout->n_q_heads, n_seqs, q, q_dtype, seq_lens,
                                     max_seq_len, block_table, kvq::to_dev(rot_k), pool, s, workspace,
                                     o_rot, err, stream, wg, kvq::to_dev(rot_v));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_decode_attention");
}

kvq_status kvq_fold_wo(int d_model, int n_q_heads, int n_kv_heads, const void* w_o, kvq_dtype w_dtype,
                       kvq_rot rot_v, void* w_folded, kvq_dtype out_dtype, kvq_stream stream) {
  if (d_model < 1 || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0)
    return fail(KVQ_EINVAL, "bad shape d_model %d n_q_heads %d n_kv_heads %d", d_model, n_q_heads, n_kv_heads);
  if (!valid_dtype(w_dtype) || !valid_dtype(out_dtype)) return fail(KVQ_EINVAL, "bad dtype");
  KVQ_CHECK(check_rot(rot_v, "rot_v"));
  KVQ_PTR(w_o, "w_o");
  KVQ_PTR(w_folded, "w_folded");
  if (w_o == w_folded) return fail(KVQ_EINVAL, "w_o and w_folded must not alias");
  cudaError_t e = kvq::launch_fold_wo(d_model, n_q_heads, n_q_heads / n_kv_heads, w_o, w_dtype,
                                      kvq::to_dev(rot_v), w_folded, out_dtype, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_fold_wo");
}

kvq_status kvq_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                        kvq_dtype w_dtype, float* y, kvq_stream stream) {
  if (n_rows < 0 || d_model < 1 || k_dim < 1)
    return fail(KVQ_EINVAL, "bad shape n_rows %d d_model %d k_dim %d", n_rows, d_model, k_dim);
  if (k_dim % 32 != 0) return fail(KVQ_EUNSUPPORTED, "k_dim %d is not a multiple of 32", k_dim);
  if (!valid_dtype(w_dtype)) return fail(KVQ_EINVAL, "bad dtype %d", (int)w_dtype);
  if (n_rows == 0) return KVQ_OK;
  KVQ_PTR(x, "x");
  KVQ_PTR(w, "w");
  KVQ_PTR(y, "y");
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  cudaError_t e = kvq::launch_out_proj(n_rows, d_model, k_dim, x, w, w_dtype, y, err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_out_proj");
}

kvq_status kvq_wo_packed_bytes(int d_model, int k_dim, size_t* bytes) {
  if (!bytes) return fail(KVQ_EINVAL, "bytes is NULL");
  if (d_model < 1 || k_dim < 1) return fail(KVQ_EINVAL, "bad shape d_model %d k_dim %d", d_model, k_dim);
  if (k_dim % 32 != 0) return fail(KVQ_EUNSUPPORTED, "k_dim %d is not a multiple of 32", k_dim);
  *bytes = kvq::wo_packed_bytes(d_model, k_dim);
  return KVQ_OK;
}

kvq_status kvq_pack_wo(int d_model, int k_dim, const void* w, void* w_packed, kvq_stream stream) {
  size_t bytes = 0;
  KVQ_CHECK(kvq_wo_packed_bytes(d_model, k_dim, &bytes));
  KVQ_PTR(w, "w");
  KVQ_PTR(w_packed, "w_packed");
  cudaError_t e = kvq::launch_pack_wo(d_model, k_dim, w, w_packed, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_pack_wo");
}

kvq_status kvq_out_proj_packed(int n_rows, int d_model, int k_dim, const float* x, const void* w_packed, float* y,
                               kvq_stream stream) {
  if (n_rows < 0 || d_model < 1 || k_dim < 1)
    return fail(KVQ_EINVAL, "bad shape n_rows %d d_model %d k_dim %d", n_rows, d_model, k_dim);
  if (k_dim % 32 != 0) return fail(KVQ_EUNSUPPORTED, "k_dim %d is not a multiple of 32", k_dim);
  if (n_rows == 0) return KVQ_OK;
  KVQ_PTR(x, "x");
  KVQ_PTR(w_packed, "w_packed");
  KVQ_PTR(y, "y");
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  cudaError_t e = kvq::launch_out_proj_packed(n_rows, d_model, k_dim, x, w_packed, y, err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_out_proj_packed");
}

kvq_status kvq_calib_workspace_size(int n_tok, int n_qpos, int n_kv_heads, int gqa, int joint,
                                    size_t* bytes) {
  if (!bytes) return fail(KVQ_EINVAL, "bytes is NULL");
  if (n_tok < 1 || n_qpos < 1 || n_qpos > n_tok || n_kv_heads < 1 || gqa < 1)
    return fail(KVQ_EINVAL, "bad shape n_tok %d n_qpos %d n_kv_heads %d gqa %d", n_tok, n_qpos, n_kv_heads, gqa);
  *bytes = kvq::calib_workspace_bytes(n_tok, n_qpos, n_kv_heads, gqa, joint ? 1 : 0);
  return KVQ_OK;
}

kvq_status kvq_calib_nmse(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model, const void* q,
                          const void* k, const void* v, kvq_dtype dtype, const void* w_o,
                          kvq_dtype w_dtype, int n_cand, const kvq_rot* cand, int n_clip,
                          const float* clips, const float* mu, int joint, double* nmse, double* ref,
                          void* workspace, size_t workspace_bytes, kvq_stream stream) {
  if (n_tok < 1 || n_qpos < 1 || n_qpos > n_tok || n_kv_heads < 1 || gqa < 1 || d_model < 1)
    return fail(KVQ_EINVAL, "bad shape n_tok %d n_qpos %d n_kv_heads %d gqa %d d_model %d", n_tok, n_qpos,
                n_kv_heads, gqa, d_model);
  if (n_tok > 12288) return fail(KVQ_EUNSUPPORTED, "n_tok %d > 12288 calibration tokens", n_tok);
  const long long gd = joint ? (long long)n_kv_heads * gqa * kvq::D : (long long)gqa * kvq::D;
  if (gd > 12288) return fail(KVQ_EUNSUPPORTED, "scored head group of %lld channels > 12288", gd);
  if (!valid_dtype(dtype) || !valid_dtype(w_dtype)) return fail(KVQ_EINVAL, "bad dtype");
  if (n_cand < 1 || !cand) return fail(KVQ_EINVAL, "need at least one candidate (host array)");
  if (n_clip < 1 || !clips) return fail(KVQ_EINVAL, "need at least one clip ratio (host array)");
  for (int i = 0; i < n_clip; ++i)
    if (!valid_clip(clips[i])) return fail(KVQ_EINVAL, "clip[%d] = %g outside (0, 1]", i, clips[i]);
  for (int i = 0; i < n_cand; ++i) {
    char name[32];
    snprintf(name, sizeof(name), "cand[%d]", i);
    KVQ_CHECK(check_rot(cand[i], name));
  }
  KVQ_PTR(q, "q");
  KVQ_PTR(k, "k");
  KVQ_PTR(v, "v");
  KVQ_PTR(w_o, "w_o");
  KVQ_PTR(nmse, "nmse");
  KVQ_PTR(ref, "ref");
  KVQ_PTR(workspace, "workspace");
  if (mu && !aligned16(mu)) return fail(KVQ_EINVAL, "mu is not 16-byte aligned");
  const size_t need = kvq::calib_workspace_bytes(n_tok, n_qpos, n_kv_heads, gqa, joint ? 1 : 0);
  if (workspace_bytes < need) return fail(KVQ_EINVAL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  cudaError_t e = kvq::launch_calib(n_tok, n_qpos, n_kv_heads, gqa, d_model, q, k, v, dtype, w_o, w_dtype,
                                    n_cand, cand, n_clip, clips, mu, joint ? 1 : 0, nmse, ref, workspace, err,
                                    stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_calib_nmse");
}

kvq_status kvq_report_workspace_size(int n_tok, int n_qpos, int n_kv_heads, int gqa, size_t* bytes) {
  if (!bytes) return fail(KVQ_EINVAL, "bytes is NULL");
  if (n_tok < 1 || n_qpos < 1 || n_qpos > n_tok || n_kv_heads < 1 || gqa < 1)
    return fail(KVQ_EINVAL, "bad shape n_tok %d n_qpos %d n_kv_heads %d gqa %d", n_tok, n_qpos, n_kv_heads, gqa);
  *bytes = kvq::report_workspace_bytes(n_tok, n_qpos, n_kv_heads, gqa);
  return KVQ_OK;
}

kvq_status kvq_head_error_report(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model, const void* q,
                                 const void* k, const void* v, kvq_dtype dtype, const void* w_o, kvq_dtype w_dtype,
                                 kvq_rot rot_k, kvq_rot rot_v, const float* mu, float clip_k, float clip_v,
                                 double* out, void* workspace, size_t workspace_bytes, kvq_stream stream) {
  if (n_tok < 1 || n_qpos < 1 || n_qpos > n_tok || n_kv_heads < 1 || d_model < 1)
    return fail(KVQ_EINVAL, "bad shape n_tok %d n_qpos %d n_kv_heads %d d_model %d", n_tok, n_qpos, n_kv_heads,
                d_model);
  if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8)
    return fail(KVQ_EUNSUPPORTED, "query heads per KV head %d: supported 1, 2, 4, 8", gqa);
  if (n_tok > 12288) return fail(KVQ_EUNSUPPORTED, "n_tok %d > 12288 calibration tokens", n_tok);
  if (!valid_dtype(dtype) || !valid_dtype(w_dtype)) return fail(KVQ_EINVAL, "bad dtype");
  if (!valid_clip(clip_k) || !valid_clip(clip_v))
    return fail(KVQ_EINVAL, "clip ratios must lie in (0, 1] (got %g, %g)", clip_k, clip_v);
  KVQ_CHECK(check_rot(rot_k, "rot_k"));
  KVQ_CHECK(check_rot(rot_v, "rot_v"));
  KVQ_PTR(q, "q");
  KVQ_PTR(k, "k");
  KVQ_PTR(v, "v");
  KVQ_PTR(w_o, "w_o");
  KVQ_PTR(out, "out");
  KVQ_PTR(workspace, "workspace");
  if (mu && !aligned16(mu)) return fail(KVQ_EINVAL, "mu is not 16-byte aligned");
  const size_t need = kvq::report_workspace_bytes(n_tok, n_qpos, n_kv_heads, gqa);
  if (workspace_bytes < need) return fail(KVQ_EINVAL, "workspace %zu bytes < %zu required", workspace_bytes, need);
  unsigned* err = nullptr;
  KVQ_CHECK(device_error_word(&err));
  cudaError_t e = kvq::launch_head_report(n_tok, n_qpos, n_kv_heads, gqa, d_model, q, k, v, dtype, w_o, w_dtype,
                                          kvq::to_dev(rot_k), kvq::to_dev(rot_v), mu, clip_k, clip_v, out,
                                          workspace, err, stream);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "kvq_head_error_report");
}

}  // extern "C"
