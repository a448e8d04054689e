/*
 * kvq.h -- C ABI of libkvq: rotated INT2 KV-cache attention on NVIDIA GB300 (sm_103a).
 *
 * The operations follow "Output-Aware Rotation for INT2 KV-Cache Quantization"
 * (OptR) and the "Output-aware INT2 KV-cache rotation evaluation" page:
 *
 *   write path   keys are centred by a per-channel mean mu (§4.1, Eq. 19), rotated
 *                per KV head (k - mu) R_K = k R_K - mu R_K (Eq. 20), values rotated
 *                v R_V (Eq. 27), then quantized per token in groups of 128 channels
 *                to 4 levels (§3.1 Eq. 4, §5 implementation details, Table A) and
 *                packed into a paged cache.
 *   read path    q is rotated once, q R_K (Eqs. 21-22, 26); scores, softmax and the
 *                value readout run straight off the packed pages; the readout stays
 *                in the rotated-V basis o' = o R_V (Eq. 27) and meets the folded
 *                W_O-bar_j = W_O,j R_V,h(j) (Eqs. 29-31) in the output projection.
 *   calibration  post-W_O NMSE (Eq. 10) of every candidate rotation x clip ratio,
 *                as in the evaluation page's candidate search.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller unless the
 *     argument says "host".  The library never allocates device memory; calls
 *     that need scratch take a caller-provided workspace sized by the matching
 *     *_workspace_size function.  Exception: the per-step activations may be
 *     pinned (page-locked, device-mapped) host memory - q, k_new and v_new of
 *     kvq_decode_attention(_win) and kvq_decode_step(_win), and y of
 *     kvq_out_proj_packed - which the kernels then read or write across the
 *     host link themselves (results identical to device buffers).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream)
 *     and performs no implicit synchronisation, except kvq_device_check.
 *   - Every tensor is dense, row-major, with the shapes given below.  Pointers
 *     must be 16-byte aligned; otherwise KVQ_EINVAL.
 *   - head_dim must be 128 (the group size of the method); anything else returns
 *     KVQ_EUNSUPPORTED.  There is no fallback path of any kind.
 *   - A non-OK status leaves outputs unspecified; kvq_last_error() returns a
 *     thread-local, human-readable reason.
 *   - Data-dependent indices that cannot be checked on the host without a
 *     synchronisation (block-table entries, sequence lengths) are bounds-checked
 *     in the kernels: an out-of-range entry is skipped and recorded in a device
 *     error word, which kvq_device_check() reads back as KVQ_EDEVICE_FLAG.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* kvq_stream;

typedef enum {
  KVQ_OK = 0,
  KVQ_EINVAL = -1,        /* bad argument: null pointer, bad shape, misalignment, bad clip */
  KVQ_EUNSUPPORTED = -2,  /* valid request outside what is implemented (head_dim != 128, ...) */
  KVQ_ECUDA = -3,         /* a CUDA runtime call failed (launch error, no device, ...) */
  KVQ_EDEVICE_FLAG = -4   /* a kernel met an out-of-range block-table entry or length */
} kvq_status;

typedef enum {
  KVQ_ROT_IDENTITY = 0,         /* R = I */
  KVQ_ROT_SIGNED_HADAMARD = 1,  /* R_h = diag(s_h) H_128 / sqrt(128), H Sylvester-ordered */
  KVQ_ROT_DENSE = 2             /* R_h given explicitly (e.g. exp(A - A^T), OptR Eq. 11) */
} kvq_rot_kind;

typedef enum {
  KVQ_F32 = 0,
  KVQ_BF16 = 1
} kvq_dtype;

/* One orthogonal rotation per KV head.  A row vector x is rotated as x R_h.
 *   signs: [n_heads][128] float, each +1 or -1       (KVQ_ROT_SIGNED_HADAMARD)
 *   dense: [n_heads][128][128] float, R_h[c][d] at c*128 + d, row = input channel
 *                                                      (KVQ_ROT_DENSE)
 * Unused pointers may be NULL. */
typedef struct {
  int kind;             /* kvq_rot_kind */
  const float* signs;
  const float* dense;
} kvq_rot;

/* Paged cache geometry.
 * The pool is uint8 [num_blocks][n_kv_heads][72 * page_tokens]: one record per
 * (physical page, KV head), laid out as
 *   [0, 32P)     K codes: token slot o at 32*o, 128 two-bit codes, channel i in
 *                byte i/4 at bits 2*(i%4)
 *   [32P, 64P)   V codes, same layout
 *   [64P, 68P)   K meta: slot o at 64P + 4*o = fp16 scale, fp16 zero
 *   [68P, 72P)   V meta
 * Position pos of sequence b lives in page block_table[b * max_blocks_per_seq + pos / P],
 * slot pos % P.  A dequantized value is zero + scale * code. */
typedef struct {
  int head_dim;            /* must be 128 */
  int page_tokens;         /* P: 8 or 16 */
  int n_kv_heads;          /* H_kv >= 1 */
  int n_q_heads;           /* H_q, a multiple of H_kv; query head j reads KV head j / (H_q/H_kv) */
  int num_blocks;          /* physical pages in the pool */
  int max_blocks_per_seq;  /* row stride of block_table */
} kvq_layout;

/* BF16 sink and recent windows ("Output-Aware Rotation for INT2 KV-Cache
 * Quantization", §5 implementation details and Table A: 64 sink and 256 recent
 * tokens stay in BF16; appendix "OptR Algorithm" and "Key-mean estimation and
 * application": window tokens skip INT2, their keys keep the centring, their
 * values stay unchanged in BF16).
 * At length L, position p < L is a window token iff p < sink_tokens or
 * p >= L - recent_tokens; the windowed decode reads it from `buf` and every
 * other position from the INT2 pages (which still hold every token).
 *   window key   = bf16_rn(fp32(k - mu))   centred, not rotated (mu NULL: k)
 *   window value = bf16_rn(v)              unchanged (a copy for bf16 inputs)
 * Neither is rotated: the windowed decode rotates the window part of its
 * readout by R_V once, so that the output stays in the rotated-V basis (Eq. 27).
 * buf: uint8 [n_seqs][n_kv_heads][(sink + recent) / 8][4096], caller-owned,
 * 16-byte aligned.  Record i of a (sequence, KV head) holds slots 8i .. 8i + 7:
 * 8 key rows, then 8 value rows, each 128 bf16 (256 bytes); position p uses
 * slot p (p < sink) or sink + p % recent; inside row r = slot % 8 the 16-byte
 * chunk c (channels 8c .. 8c + 7) is stored at chunk position c ^ r.
 * sink_tokens: a multiple of 64; recent_tokens: a multiple of 8;
 * sink_tokens + recent_tokens <= 65536.  Both 0: no windows. */
typedef struct {
  int sink_tokens;
  int recent_tokens;
  uint8_t* buf;
} kvq_window;

/* Size in bytes of the pool described by `layout`. */
size_t kvq_pool_bytes(const kvq_layout* layout);

/* Thread-local message describing the last non-OK status returned on this thread. */
const char* kvq_last_error(void);

/* Synchronise `stream`, then read and clear the device error word.
 * KVQ_OK if no kernel recorded an out-of-range index since the last check,
 * KVQ_EDEVICE_FLAG otherwise (the message names the first recorded error). */
kvq_status kvq_device_check(kvq_stream stream);

/* Key mean (OptR appendix, "Key-mean estimation and application", Eq. 19):
 *   mu[h][c] = (1/n_tok) sum_t k[t][h][c]
 * k: [n_tok][n_kv_heads][128] of dtype; mu: [n_kv_heads][128] float (written). */
kvq_status kvq_key_mean(int n_tok, int n_kv_heads, const void* k, kvq_dtype dtype,
                        float* mu, kvq_stream stream);

/* Per-head rotation of row vectors (Eq. 20's precomputed mu R_K; Eq. 22's q R_K):
 *   y[r][j] = x[r][j] R_{j / heads_per_rot}
 * x, y: [n_rows][n_heads][128] float (may not alias); rot covers
 * n_heads / heads_per_rot heads. */
kvq_status kvq_rotate_heads(int n_rows, int n_heads, int heads_per_rot, const float* x,
                            kvq_rot rot, float* y, kvq_stream stream);

/* Quantize-append (OptR §6 "Efficiency Analysis" cache-write kernel; Eqs. 4, 20, 21, 27):
 * for every new token t of sequence b at position pos = start_pos[b] + (t - cu_new[b]),
 * and every KV head h,
 *   x_K = k[t][h] R_K,h - mu_rot_k[h]      (= (k - mu) R_K; mu_rot_k NULL means mu = 0)
 *   x_V = v[t][h] R_V,h
 * each x is quantized as one group of 128: lo = c*min(x), hi = c*max(x),
 * scale = fp16_rn((hi - lo)/3), zero = fp16_rn(lo),
 * code = clamp(rint((x - zero)/scale), 0, 3) (code 0 where scale == 0),
 * and written to the token's page slot (see kvq_layout).
 *   k, v:        [n_new_total][n_kv_heads][128] of dtype
 *   cu_new:      int32 [n_seqs + 1], cu_new[0] = 0, non-decreasing, cu_new[n_seqs] = n_new_total
 *   start_pos:   int32 [n_seqs]
 *   block_table: int32 [n_seqs][max_blocks_per_seq]
 *   mu_rot_k:    float [n_kv_heads][128] or NULL
 *   clip_k, clip_v in (0, 1]
 *   pool:        uint8, kvq_pool_bytes(layout) bytes, written in place
 * Pages referenced by an out-of-range block-table entry or position are skipped
 * and flagged (kvq_device_check). */
kvq_status kvq_quantize_append(const kvq_layout* layout, int n_seqs, int n_new_total,
                               const void* k, const void* v, kvq_dtype dtype,
                               const int32_t* cu_new, const int32_t* start_pos,
                               const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v,
                               const float* mu_rot_k, float clip_k, float clip_v,
                               uint8_t* pool, kvq_stream stream);

/* Workspace bytes needed by kvq_decode_attention for this many sequences and
 * work partitions (n_splits = 0: the count the library would choose for
 * max_seq_len).  Computed on the host from the arguments alone. */
kvq_status kvq_decode_workspace_size(const kvq_layout* layout, int n_seqs, int max_seq_len,
                                     int n_splits, size_t* bytes);

/* Split-K decode attention straight off the packed cache (OptR Eqs. 1-2, 5, 22, 26, 27):
 * for sequence b and query head j with KV head h = j / (H_q / H_kv),
 *   q'_j   = q[b][j] R_K,h
 *   a_s    = q'_j . (zero_s + scale_s * codeK_s) / sqrt(128),   s < seq_lens[b]
 *   p      = softmax(a)
 *   o_rot[b][j] = sum_s p_s (zero_s + scale_s * codeV_s)      (rotated-V basis)
 * The cached tokens of the batch, taken as one list of (sequence, KV head,
 * 32-token chunk) entries, are cut into 4 * n_splits equal contiguous slices,
 * one per warp (n_splits work partitions of 4 warps; 0 = the library's choice,
 * one full wave of the GPU, which runs as one thread block per SM; other
 * counts run as n_splits blocks of 4 warps).  Each slice yields a partial
 * softmax per (sequence, KV head) it
 * touches, and the partials of a unit are merged by a log-sum-exp combine in
 * slice order, so the result does not depend on timing.  A sequence of
 * length 0 yields a zero vector.  Out-of-range lengths or block ids are
 * flagged (kvq_device_check) and the affected outputs are unspecified.
 *   q:       [n_seqs][n_q_heads][128] of q_dtype
 *   seq_lens int32 [n_seqs]; max_seq_len (host) >= every seq_lens[b];
 *            n_seqs <= 65535 and n_seqs * n_kv_heads * ceil(max_seq_len / 32) < 2^30
 *   o_rot:   float [n_seqs][n_q_heads][128] (written)
 *   workspace: >= kvq_decode_workspace_size bytes, 16-byte aligned. */
kvq_status kvq_decode_attention(const kvq_layout* layout, int n_seqs, const void* q,
                                kvq_dtype q_dtype, const int32_t* seq_lens, int max_seq_len,
                                const int32_t* block_table, kvq_rot rot_k, const uint8_t* pool,
                                int n_splits, void* workspace, size_t workspace_bytes,
                                float* o_rot, kvq_stream stream);

/* One decode step: the quantize-append of each sequence's new token fused with
 * the decode attention that reads it ("Output-Aware Rotation for INT2 KV-Cache
 * Quantization", §6 "Efficiency Analysis": the cache-write kernel and the decode
 * of the rotated INT2 pipeline; Eqs. 4, 20-22, 26, 27).  For every sequence b
 * with seq_lens[b] >= 1 the token at position seq_lens[b] - 1 is written as
 * kvq_quantize_append would write it (k_new[b], v_new[b]; same rotations, key
 * shift and clip ratios, the same bytes), and then o_rot is what
 * kvq_decode_attention returns over seq_lens[b] tokens.  A sequence of length 0
 * appends nothing and yields a zero vector.  The query preparation writes the
 * new tokens, and the decode kernel reads their pages only after it, so the
 * step is one call with no separate append launch.
 *   q:            [n_seqs][n_q_heads][128] of dtype
 *   k_new, v_new: [n_seqs][n_kv_heads][128] of dtype
 *   mu_rot_k:     float [n_kv_heads][128] (mu R_K) or NULL; clip_k, clip_v in (0, 1]
 *   pool:         written in place (the new tokens' slots) and read
 *   workspace:    >= kvq_decode_workspace_size bytes
 * Other arguments, limits and errors as kvq_decode_attention and
 * kvq_quantize_append (an out-of-range block id is skipped and flagged). */
kvq_status kvq_decode_step(const kvq_layout* layout, int n_seqs, const void* q, const void* k_new,
                           const void* v_new, kvq_dtype dtype, const int32_t* seq_lens, int max_seq_len,
                           const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v,
                           const float* mu_rot_k, float clip_k, float clip_v, uint8_t* pool,
                           int n_splits, void* workspace, size_t workspace_bytes, float* o_rot,
                           kvq_stream stream);

/* Window copies of appended tokens (see kvq_window).  For every new token of
 * sequence b at position p = start_pos[b] + (t - cu_new[b]) that is a window
 * token at the sequence's new length (p < sink, or p >= start_pos[b] + n_new_b -
 * recent), and every KV head h, writes bf16_rn(fp32(k - mu_k[h])) and
 * bf16_rn(v) into its slot.  Call it beside kvq_quantize_append with the same
 * tokens.
 *   k, v, dtype, cu_new, start_pos: as in kvq_quantize_append
 *   mu_k:  float [n_kv_heads][128], the UNROTATED key mean, or NULL
 *   win:   host struct; buf rows are indexed by the sequence index b */
kvq_status kvq_window_append(const kvq_layout* layout, int n_seqs, int n_new_total, const void* k,
                             const void* v, kvq_dtype dtype, const int32_t* cu_new,
                             const int32_t* start_pos, const float* mu_k, const kvq_window* win,
                             kvq_stream stream);

/* Workspace bytes of kvq_decode_attention_win: kvq_decode_workspace_size plus,
 * with windows, a second set of partials, the windows' query fragments and spans. */
kvq_status kvq_decode_workspace_size_win(const kvq_layout* layout, int n_seqs, int max_seq_len,
                                         int n_splits, const kvq_window* win, size_t* bytes);

/* Decode attention over INT2 pages and BF16 windows together (OptR Eqs. 1-2,
 * 5, 22, 24, 26, 27 with the windows of kvq_window): one softmax over
 *   a_s = q'_j . (zero_s + scale_s * codeK_s) / sqrt(128)   INT2 positions (q' = q R_K)
 *   a_s = q_j . key~_s / sqrt(128)                          window positions (unrotated q)
 *   o_rot[b][j] = sum_INT2 p_s (zero_s + scale_s * codeV_s) + (sum_window p_s value~_s) R_V,h
 * (rotated-V basis; the window values are stored unrotated, so their part of
 * the readout is rotated once, in fp32, per sequence and query head).
 * The INT2 positions of the batch are split across the warps of the grid as in
 * kvq_decode_attention, the 8-token window records in a second equal split;
 * each split yields its own partials and the combine merges both in a fixed
 * order (deterministic).  win NULL, or both window sizes 0, is
 * kvq_decode_attention (rot_v unused).  Arguments otherwise as
 * kvq_decode_attention; the workspace must hold kvq_decode_workspace_size_win bytes. */
kvq_status kvq_decode_attention_win(const kvq_layout* layout, int n_seqs, const void* q,
                                    kvq_dtype q_dtype, const int32_t* seq_lens, int max_seq_len,
                                    const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v,
                                    const uint8_t* pool, const kvq_window* win, int n_splits,
                                    void* workspace, size_t workspace_bytes, float* o_rot,
                                    kvq_stream stream);

/* One decode step with BF16 sink / recent windows: kvq_decode_step's fused
 * append and decode, plus the new token's window copy ("Output-Aware Rotation
 * for INT2 KV-Cache Quantization", §5 implementation details, Table A; §6 the
 * cache-write kernel and decode).  For every sequence with seq_lens[b] >= 1 the
 * token at position seq_lens[b] - 1 is written to the pool as kvq_quantize_append
 * would write it and to the windows as kvq_window_append would (key k - mu_k,
 * value v, both bf16; sink slot if the position is below sink_tokens, else the
 * recent ring), and o_rot is then what kvq_decode_attention_win returns over
 * seq_lens[b] tokens.  One call: the query preparation writes both, and the
 * decode reads them only after it.
 *   mu_k:      float [n_kv_heads][128] unrotated key mean for the window keys, or NULL
 *   win:       the windows (written in place and read); sink + recent may be 0
 *   workspace: >= kvq_decode_workspace_size_win bytes
 * Other arguments, limits and errors as kvq_decode_step and kvq_decode_attention_win. */
kvq_status kvq_decode_step_win(const kvq_layout* layout, int n_seqs, const void* q, const void* k_new,
                               const void* v_new, kvq_dtype dtype, const int32_t* seq_lens, int max_seq_len,
                               const int32_t* block_table, kvq_rot rot_k, kvq_rot rot_v, const float* mu_rot_k,
                               const float* mu_k, float clip_k, float clip_v, uint8_t* pool, const kvq_window* win,
                               int n_splits, void* workspace, size_t workspace_bytes, float* o_rot,
                               kvq_stream stream);

/* The same decode attention for callers that cannot allocate device memory
 * (the paper has no counterpart; this is a deployment convenience).
 * Serving engines that reserve all device memory up front and forbid allocation
 * while requests are in flight, and host frameworks that hand a plugin only the
 * tensors it reads and writes, cannot provide kvq_decode_attention's workspace.
 * This variant keeps the split partials in a fixed 4 MiB buffer inside the
 * library (a __device__ array that every GPU loading the library holds until
 * process exit) and allocates nothing.
 *   - Arguments are those of kvq_decode_attention without the workspace.
 *   - With n_splits = 0 it takes the largest number of work partitions, up
 *     to the library's choice, whose partials fit in the buffer.  If the
 *     partials still need more than 4 MiB (kvq_decode_workspace_size), or an
 *     explicit n_splits needs more, it returns KVQ_EUNSUPPORTED with a
 *     message naming both sizes.
 *   - The first call on each device looks up the buffer's device address; make
 *     that first call, with the device current, before any stream capture.
 *     `stream` must belong to the current device, and the looked-up address
 *     does not survive a cudaDeviceReset of that device.
 *   - All calls share the buffer: calls that overlap on the GPU (other streams,
 *     other host threads) race and must be serialised by the caller.  Each call
 *     writes every byte of scratch it reads, so nothing needs clearing. */
kvq_status kvq_decode_attention_noalloc(const kvq_layout* layout, int n_seqs, const void* q,
                                        kvq_dtype q_dtype, const int32_t* seq_lens, int max_seq_len,
                                        const int32_t* block_table, kvq_rot rot_k,
                                        const uint8_t* pool, int n_splits, float* o_rot,
                                        kvq_stream stream);

/* W_O folding (OptR Eqs. 29-31): for query head j with KV head h = j / (H_q / H_kv),
 *   w_folded[:, j*128:(j+1)*128] = w_o[:, j*128:(j+1)*128] R_V,h
 * w_o: [d_model][n_q_heads*128] of w_dtype; w_folded: same shape, out_dtype
 * (bf16 output is rounded to nearest even). */
kvq_status kvq_fold_wo(int d_model, int n_q_heads, int n_kv_heads, const void* w_o,
                       kvq_dtype w_dtype, kvq_rot rot_v, void* w_folded, kvq_dtype out_dtype,
                       kvq_stream stream);

/* Output projection (OptR Eqs. 3, 7, 31): y[r] = sum_k x[r][k] w[n][k] for n < d_model,
 * i.e. y = x W^T with x = o_rot viewed as [n_rows][n_q_heads*128] and W = the folded W_O.
 *   x: float [n_rows][k_dim]; w: [d_model][k_dim] of w_dtype; y: float [n_rows][d_model].
 * k_dim must be a multiple of 32 (it is n_q_heads * 128); otherwise KVQ_EUNSUPPORTED.
 * Tensor-core products with fp32 accumulation: x enters as a bf16 high part plus a bf16
 * remainder (about 16 significant bits), an fp32 w as two bf16 parts likewise; partial sums
 * over K are added in a fixed order, so the result does not depend on timing. */
kvq_status kvq_out_proj(int n_rows, int d_model, int k_dim, const float* x, const void* w,
                        kvq_dtype w_dtype, float* y, kvq_stream stream);

/* The folded W_O in the box order of the projection (the same product as kvq_out_proj with
 * a bf16 W, for decode-size batches where the weight stream is the cost): W (bf16
 * [d_model][k_dim], e.g. kvq_fold_wo's output) is stored as one contiguous 16 KB block per
 * (128-row tile T, 64-column stage c), at (T * ceil(k_dim / 64) + c) * 16 KB; inside a block,
 * row r (0..127) occupies 128 bytes at r * 128, holding columns 64 c .. 64 c + 63 as eight
 * 16-byte chunks, chunk j stored at position j ^ (r % 8) (rows past d_model and columns past
 * k_dim are zero).  Each block is then one bulk copy straight into the tensor cores' operand
 * layout, one DRAM stream per block instead of 128 rows of 128 bytes.
 * k_dim must be a multiple of 32 (KVQ_EUNSUPPORTED otherwise). */
kvq_status kvq_wo_packed_bytes(int d_model, int k_dim, size_t* bytes);
kvq_status kvq_pack_wo(int d_model, int k_dim, const void* w, void* w_packed, kvq_stream stream);

/* kvq_out_proj with w = the packed W of kvq_pack_wo (bf16): y = x W^T, the same tensor-core
 * arithmetic and summation order as kvq_out_proj with the row-major bf16 W (equal results).
 * The packed W is a static weight: the projection starts streaming it while the preceding
 * kernel on the stream (e.g. the decode's combine) still runs, so w_packed must have been
 * written before that kernel began (kvq_pack_wo once at set-up; not by the kernel launched
 * immediately before this call).  x may come from the preceding kernel. */
kvq_status kvq_out_proj_packed(int n_rows, int d_model, int k_dim, const float* x, const void* w_packed, float* y,
                               kvq_stream stream);

/* Workspace bytes for kvq_calib_nmse. */
kvq_status kvq_calib_workspace_size(int n_tok, int n_qpos, int n_kv_heads, int gqa, int joint,
                                    size_t* bytes);

/* Candidate x clip sweep scored by post-W_O NMSE ("Output-aware INT2 KV-cache rotation
 * evaluation": candidate search on calibration queries; OptR Eq. 10 and the appendix
 * calibration details: final query positions, per-KV-head selection).
 * For candidate i (rotation R_i applied to the keys and values of every head) and
 * clip ratio c (applied to both):
 *   keys  k~ = Q_2((k - mu) R_i; c) (mu NULL: no centring),  values v~ = Q_2(v R_i; c)
 *   queries at positions t = n_tok - n_qpos .. n_tok - 1, causal (s <= t), rotated by R_i
 *   o~'   = attention readout (rotated basis), y~_h = sum_{j in G_h} o~'_j (W_O,j R_i)^T
 *   y_h   = the same with unquantized, unrotated, uncentred k, v
 *   nmse[i][c][h] = sum_t ||y~_h - y_h||^2 / ref[h],  ref[h] = sum_t ||y_h||^2
 * With joint != 0 the outputs are summed over KV heads before the norms (one column).
 *   q: [n_qpos][n_kv_heads*gqa][128]; k, v: [n_tok][n_kv_heads][128]   (dtype)
 *   w_o: [d_model][n_kv_heads*gqa*128] (w_dtype, unfolded)
 *   cand: HOST array of n_cand rotations (their signs/dense pointers are device pointers)
 *   clips: HOST array of n_clip ratios in (0, 1]
 *   mu: float [n_kv_heads][128] or NULL
 *   nmse: double [n_cand][n_clip][joint ? 1 : n_kv_heads]; ref: double [joint ? 1 : n_kv_heads]
 *   workspace: >= kvq_calib_workspace_size bytes.
 * The quantizer's decisions are exact (double-float rotation, as the cache write); each
 * candidate's attention is computed by the decode kernels over a page pool of the
 * quantized trace, one sequence per query position (its causal prefix), so it is scored
 * with the arithmetic the cache is read with; the reference attention runs in fp32.
 * gqa must be 1, 2, 4 or 8.  Out-of-range data found on the device sets the error word
 * (kvq_device_check).  Selection (argmin) is left to the caller. */
kvq_status kvq_calib_nmse(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model,
                          const void* q, const void* k, const void* v, kvq_dtype dtype,
                          const void* w_o, kvq_dtype w_dtype, int n_cand, const kvq_rot* cand,
                          int n_clip, const float* clips, const float* mu, int joint,
                          double* nmse, double* ref, void* workspace, size_t workspace_bytes,
                          kvq_stream stream);

/* Workspace bytes for kvq_head_error_report. */
kvq_status kvq_report_workspace_size(int n_tok, int n_qpos, int n_kv_heads, int gqa, size_t* bytes);

/* Per-head output-error report ("Output-Aware Rotation for INT2 KV-Cache
 * Quantization", Figure 5 and the appendix "Output-space error"; the key/value
 * split of Eq. 8).  For the queries at the last n_qpos positions of an n_tok-token
 * trace (causal, s <= t) and every query head j, with KV head h = j / gqa,
 *   Delta y_{t,j} = (p~^T V~ - p^T V) W_O,j^T
 * where p uses the raw keys, p~ the candidate's effective keys (centred by mu,
 * rotated by R_K, INT2 with clip_k, met by q R_K), V~ = Q_2(V R_V; clip_v) R_V^T.
 * out (device, double [5][n_kv_heads]) receives per KV head h, summed over the
 * positions and the query heads of h:
 *   [0] E       = sum ||Delta y||^2
 *   [1] E_key   = sum ||(p~ - p)^T V W_O,j^T||^2        (key-induced term of Eq. 8)
 *   [2] E_val   = sum ||p~^T (V~ - V) W_O,j^T||^2       (value-induced term)
 *   [3] E_naive = E of plain per-group INT2: identity rotations, no centring, same clips
 *   [4] Y       = sum ||p^T V W_O,j^T||^2
 * The RMS error as a percentage of plain INT2 is 100 sqrt(E / E_naive).
 * Shapes and limits as kvq_calib_nmse: q [n_qpos][n_kv_heads*gqa][128],
 * k, v [n_tok][n_kv_heads][128] (dtype), w_o [d_model][n_kv_heads*gqa*128] (w_dtype,
 * unfolded), mu float [n_kv_heads][128] (unrotated) or NULL, n_tok <= 12288.
 * Sums are in a fixed order except for d_model <= 128 (double atomics). */
kvq_status kvq_head_error_report(int n_tok, int n_qpos, int n_kv_heads, int gqa, int d_model,
                                 const void* q, const void* k, const void* v, kvq_dtype dtype,
                                 const void* w_o, kvq_dtype w_dtype, kvq_rot rot_k, kvq_rot rot_v,
                                 const float* mu, float clip_k, float clip_v, double* out,
                                 void* workspace, size_t workspace_bytes, kvq_stream stream);

/* ---- OptR gradient calibration of one KV head ("Output-Aware Rotation for INT2
 * KV-Cache Quantization", §4.2 Eq. 11, §4.3 Eqs. 12-14, §4.4 Eqs. 15-16, §4.5
 * Eqs. 17-18, Algorithm 1; §5 implementation details: lambda_K = 1, 80 Adam
 * steps at learning rate 0.02, selection every 20 steps).
 * A trace of the head: the queries of its last n_qpos positions (causal: position
 * t = n_tok - n_qpos + i attends s <= t) and its n_tok keys and values, fp32:
 *   q [n_qpos][gqa][128], k [n_tok][128], v [n_tok][128]; 1 <= n_tok <= 8192.
 * w_o: fp32 [d_model][gqa * 128], the W_O columns of the head's query heads
 * (d_model <= 8192); mu: fp32 [128], the head's (unrotated) key mean, or NULL.
 * Rotations and generators are fp64 [128][128] row-major (x R for a row x).
 * All arithmetic is fp64; Q_2's decisions (fp16 scale and zero, codes) follow
 * kvq_quantize_append's definition with the clip ratio of the role.
 * The straight-through estimator passes a channel's gradient iff it lies in its
 * group's clip range [c min, c max] (scale and zero held constant). */
typedef struct {
  const float* q;
  const float* k;
  const float* v;
  int n_tok;
  int n_qpos;
} kvq_optr_trace;

typedef enum { KVQ_OPTR_KEYS = 0, KVQ_OPTR_VALUES = 1 } kvq_optr_phase;

/* Workspace bytes for a training trace and an optional held-out trace (0, 0 if none). */
kvq_status kvq_optr_workspace_size(int n_tok, int n_qpos, int n_tok_heldout, int n_qpos_heldout, int gqa,
                                   size_t* bytes);

/* One objective and its gradient at R = r0 exp(a - a^T):
 *   KVQ_OPTR_KEYS:   L_K = mean over (t, j) of KL(p_t || p^K_t) + lambda_k ||e_K||^2 / d_model
 *                    (Eqs. 12-14; p from the raw keys, p^K from Q_2((k - mu) R; clip_k) R^T)
 *   KVQ_OPTR_VALUES: L_V = mean over (t, j) of ||e_V||^2 / d_model (Eqs. 15-16; the weights p^K
 *                    from the selected key rotation r_k_sel with clip_k, V~ = Q_2(v R; clip_v) R^T)
 * loss: device double (written); grad: device double [128][128] = dL/da, or NULL for the loss only.
 * workspace: >= kvq_optr_workspace_size(n_tok, n_qpos, 0, 0, gqa) bytes. */
kvq_status kvq_optr_loss_grad(int phase, const kvq_optr_trace* trace, int gqa, int d_model, const float* w_o,
                              const float* mu, const double* r0, const double* a, const double* r_k_sel,
                              float clip_k, float clip_v, float lambda_k, double* loss, double* grad,
                              void* workspace, size_t workspace_bytes, kvq_stream stream);

/* Algorithm 1 for one KV head: `steps` Adam steps (beta 0.9 / 0.999, eps 1e-8, rate lr)
 * on A_K from 0 for L_K, then `steps` on A_V for L_V under the selected key path.  In
 * each phase the iterate at step 0 and after every `every` steps (0: none) is a
 * candidate, scored by the same loss on `heldout` (or on `train` when NULL); the
 * lowest score wins, ties to the earlier step.
 *   r_k = r_k0 exp(A_K* - A_K*^T), r_v = r_v0 exp(A_V* - A_V*^T): device double [128][128]
 *   loss_k, loss_v: device double [steps], the training loss before each step, or NULL
 * workspace: >= kvq_optr_workspace_size(train sizes, heldout sizes, gqa) bytes.
 * The call enqueues its kernels on `stream` and returns; a generator whose norm
 * is too large for the exponential's scaling is flagged (kvq_device_check). */
kvq_status kvq_optr_calibrate_head(const kvq_optr_trace* train, const kvq_optr_trace* heldout, int gqa, int d_model,
                                   const float* w_o, const float* mu, const double* r_k0, const double* r_v0,
                                   float clip_k, float clip_v, float lambda_k, int steps, float lr, int every,
                                   double* r_k, double* r_v, double* loss_k, double* loss_v, void* workspace,
                                   size_t workspace_bytes, kvq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
