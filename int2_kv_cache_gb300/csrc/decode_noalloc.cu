// kvq_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// kvq_decode_attention keeps its split partials in a workspace that the caller
// allocates.  Some callers cannot do that: serving engines that reserve all of
// their device memory up front and forbid allocation while a request is in
// flight (a cudaMalloc can synchronise the device and fail under
// fragmentation), and host frameworks that hand a plugin only the tensors it
// reads and writes.  This entry point keeps the partials in a fixed buffer that
// belongs to the library instead.
//
// The buffer is a file-scope __device__ array of NOALLOC_SCRATCH_BYTES, so every
// GPU that loads the library holds it until the process exits.  Its device
// address is looked up once per device, on the first call made while that
// device is current; make that first call before any stream capture.  The
// stream passed in must belong to the current device, and the cached address
// does not survive a cudaDeviceReset of that device.  All calls
// share the one buffer: calls whose executions overlap on the GPU (different
// streams, or different host threads) race on it and must be serialised by the
// caller.  Every call writes all of the scratch it reads, so nothing has to be
// cleared between calls.
#include <cstdio>
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[NOALLOC_MAX_DEVICES] = {nullptr};

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_layout* layout, int n_seqs, const void* q,
                                                   kvq_dtype q_dtype, const int32_t* seq_lens,
                                                   int max_seq_len, const int32_t* block_table,
                                                   kvq_rot rot_k, const uint8_t* pool, int n_splits,
                                                   float* o_rot, kvq_stream stream) {
  size_t need = 0;
  kvq_status st = kvq_decode_workspace_size(layout, n_seqs, max_seq_len, n_splits, &need);
  if (st != KVQ_OK) return st;
  if (n_splits == 0 && need > NOALLOC_SCRATCH_BYTES) {
    // The library's choice of work partitions needs more than the buffer: take the
    // largest count below it that fits.  The workspace grows with the count, so a
    // binary search over [1, auto) finds it (if even one partition does not fit,
    // the request is refused below).
    int lo = 1, hi = kvq::decode_auto_ctas(n_seqs, layout->n_kv_heads, layout->n_q_heads / layout->n_kv_heads,
                                           max_seq_len) - 1;
    int best = 1;
    while (lo <= hi) {
      const int mid = lo + (hi - lo) / 2;
      size_t b = 0;
      st = kvq_decode_workspace_size(layout, n_seqs, max_seq_len, mid, &b);
      if (st != KVQ_OK) return st;
      if (b <= NOALLOC_SCRATCH_BYTES) {
        best = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    n_splits = best;
    st = kvq_decode_workspace_size(layout, n_seqs, max_seq_len, n_splits, &need);
    if (st != KVQ_OK) return st;
  }
  char msg[256];
  if (need > NOALLOC_SCRATCH_BYTES) {
    snprintf(msg, sizeof(msg),
             "kvq_decode_attention_noalloc: %zu bytes of split partials needed, the built-in scratch "
             "holds %zu; use fewer sequences or splits, or kvq_decode_attention with a workspace",
             need, NOALLOC_SCRATCH_BYTES);
    return kvq::set_error(KVQ_EUNSUPPORTED, msg);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::set_error(KVQ_ECUDA, "kvq_decode_attention_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES)
    return kvq::set_error(KVQ_EUNSUPPORTED, "kvq_decode_attention_noalloc: device ordinal out of range");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        snprintf(msg, sizeof(msg), "kvq_decode_attention_noalloc: cudaGetSymbolAddress failed (%s)",
                 cudaGetErrorString(e));
        return kvq::set_error(KVQ_ECUDA, msg);
      }
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  return kvq_decode_attention(layout, n_seqs, q, q_dtype, seq_lens, max_seq_len, block_table, rot_k, pool,
                              n_splits, scratch, NOALLOC_SCRATCH_BYTES, o_rot, stream);
}
