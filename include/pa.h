/*
 * pa.h -- C ABI of libpa: attention over a paged KV cache for one
 * continuous-batching step, on one GB300 (sm_103a).
 *
 * The operations follow these pages on vLLM-style serving:
 *  [TC] "vLLM中如何实现大模型推理加速技术？" (cloud.tencent.com.cn article
 *       2589754): concatenated varlen prefill (31/29/30 -> 90 tokens),
 *       continuous batching with per-op AttentionMeta, chunked prefill whose
 *       mask is offset by the cached context, prefix-cache hits whose
 *       positions start after the hit, speculative verify (1 + N tokens).
 *  [CH] "11. 推理加速(一):vLLM 原理" (chuoer47.github.io), §11.2 PagedAttention:
 *       fixed-size blocks, one block table per request, shared read-only
 *       blocks; §11.3: decode is memory-bound, prefill compute-bound.
 *  [AI] 2048ai.net page on the vLLM V1 engine, §02 推理优化 › 1. 级联推理
 *       (Cascade Inference): shared-prefix state and unique-suffix state
 *       combined by an associative, commutative merge operator.
 *
 * Conventions shared by every call
 *  - All array arguments are DEVICE pointers unless stated otherwise.  The
 *    caller owns all memory, including the workspace; no call allocates
 *    device memory or synchronises the stream (pa_read_device_status is the
 *    one exception: it reads back a status word).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All work is enqueued on it, in call order.
 *  - Element type of q, k, v, caches and outputs is bf16 (raw 16-bit
 *    patterns); lse values are fp32 natural-log sums of exp of the scaled
 *    scores.  Supported head_dim: 64 or 128.  block_size: a multiple of 16,
 *    at most 256.  num_q_heads must be a multiple of num_kv_heads; q head h
 *    reads kv head h / (num_q_heads / num_kv_heads).
 *  - Return codes: PA_OK, or an error code for bad scalar arguments, an
 *    unsupported shape, a workspace that is too small, or a CUDA launch
 *    error.  Contents of device arrays are not checked on the host (that
 *    would need a copy); kernels clamp out-of-range indices, never trap,
 *    and OR a PA_DEV_* bit into a per-device status word.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* a scalar argument or pointer is invalid   */
    PA_ERR_UNSUPPORTED = 2,   /* head_dim / block_size / grouping not built */
    PA_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than required   */
    PA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed      */
    PA_ERR_BAD_METADATA = 5   /* pa_validate_metadata found a problem      */
};

/* Bits of the per-device status word (pa_read_device_status). */
#define PA_DEV_BAD_METADATA  0x1u  /* seq_len != context_len + q_len, or qsl decreasing   */
#define PA_DEV_BAD_BLOCK     0x2u  /* a block id outside [0, num_blocks) was clamped       */
#define PA_DEV_BAD_SLOT      0x4u  /* a slot outside the pool: that row was not written    */
#define PA_DEV_WAIT_TIMEOUT  0x8u  /* a pipeline wait ran out; the kernel stopped early    */
#define PA_DEV_PLAN_OVERFLOW 0x10u /* work did not fit the workspace's item capacity       */

/* Element type of a KV pool (pa_kv_desc.kv_dtype). */
enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 };

/*
 * The paged KV pool ([CH] §11.2): two arrays (K and V) of physical blocks,
 * each [num_blocks][num_kv_heads][block_size][head_dim], row-major, so one
 * (block, kv head) is block_size*head_dim contiguous elements.  Slot s holds
 * token offset s % block_size of physical block s / block_size.  Both
 * pointers must be 16-byte aligned.
 *
 * kv_dtype PA_KV_BF16 (0, the default of a zeroed descriptor): bf16
 * elements; k_scale / v_scale are ignored.
 *
 * kv_dtype PA_KV_FP8_E4M3: quantised KV cache (2048ai.net page on the vLLM V1
 * engine, §02 推理优化: quantisation of the KV cache).  Elements are one-byte
 * OCP FP8 E4M3 codes (bias 7, 3 mantissa bits, no infinity, largest finite
 * 448, S.1111.111 = NaN); k_scale and v_scale are device fp32
 * [num_kv_heads], and an element of kv head h stands for code * k_scale[h]
 * (v_scale[h] for V).  The scales are the caller's; they must be finite and
 * positive.  head_dim must be 128.  Attention over an fp8 pool computes q in
 * f16 (|q| must stay below 65504), K and V as decoded exactly to f16 and
 * scaled in fp32 on the split-KV kernel.  Requests with q_len * group > 64
 * run on the tensor-core kernel over a bf16 copy of their blocks when the
 * workspace has room for it (pa_fp8_staging_bytes), and on the split-KV
 * kernel in pieces of 64 / group query tokens otherwise.
 * pa_prefix_attention and pa_cascade_decode decode the shared prefix's
 * blocks into a bf16 staging copy in the workspace for their tensor-core
 * prefix pass (see pa_cascade_fp8_staging_bytes); cascade decode's suffix
 * pass runs on the fp8 split-KV kernel.
 */
typedef struct pa_kv_desc {
    void *k_cache;
    void *v_cache;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t kv_dtype;       /* PA_KV_BF16 or PA_KV_FP8_E4M3 */
    int32_t reserved;       /* must be 0 */
    const float *k_scale;   /* fp8 only: device fp32 [num_kv_heads] */
    const float *v_scale;   /* fp8 only: device fp32 [num_kv_heads] */
} pa_kv_desc;

/*
 * reshape_and_cache: scatter this step's new K/V rows into their slots.
 * For every token t with s = slot_mapping[t] >= 0 and every kv head h:
 *   k_cache[s / bs][h][s % bs][:] = k[t][h][:]   (same for v)
 * bf16 pool: bit-exact copy.  fp8 pool: each element x becomes
 * e4m3(x / k_scale[h]) (v_scale for v): the quotient in IEEE binary32,
 * rounded to nearest even, then rounded to the nearest e4m3 value (ties to
 * the even mantissa), magnitudes beyond 448 saturating to 448 (NaN stays
 * NaN).  Negative slots are skipped (padding).  A slot beyond the pool is
 * skipped and flags PA_DEV_BAD_SLOT.  Duplicate slots in one call are
 * invalid (which write wins is unspecified).
 *   k, v          bf16 [num_tokens][num_kv_heads][head_dim], 16-B aligned
 *   slot_mapping  int64 [num_tokens]
 * Source: [CH] §11.2 (tokens fill fixed-size blocks allocated on demand);
 * the operation name comes from vLLM's cache-write kernel.
 */
int pa_write_kv(const void *k, const void *v, const int64_t *slot_mapping, int32_t num_tokens,
                const pa_kv_desc *kv, void *stream);

/*
 * Workspace bytes pa_attention / pa_attention_ex need for a step with these
 * sizes (independent of the lengths in the metadata).  The workspace holds
 * the device-built work list, split-KV partial states and completion
 * counters; it must be 256-byte aligned and stay untouched while the call's
 * kernels run.  Returns 0 for invalid sizes.
 */
size_t pa_attention_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim);

/*
 * Extra workspace bytes, on top of pa_attention_workspace_size, that let an
 * fp8 (e4m3) pool run its long requests (q_len * group > 64) on the
 * tensor-core kernel: num_blocks bf16 blocks of K and of V, i.e. the blocks
 * of the step's long requests (sum of ceil(seq_len / block_size)).  Any
 * workspace beyond the step's own layout serves as this staging area;
 * pa_attention decodes the long requests' blocks into it (exactly: every
 * e4m3 value is a bf16 value; the scales stay separate) in request order
 * while they fit, and runs the rest as split-KV pieces.  Returns 0 for
 * invalid sizes.  bf16 pools ignore any extra workspace.
 */
size_t pa_fp8_staging_bytes(int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int64_t num_blocks);

/*
 * Varlen paged attention for one continuous-batching step ([TC], [CH]).
 * Request b owns query tokens [qsl[b], qsl[b+1]) (qsl = query_start_loc,
 * int32 [num_seqs+1], qsl[0] = 0, non-decreasing, qsl[num_seqs] <=
 * num_q_tokens; query rows from qsl[num_seqs] on belong to no request and
 * out / lse there are left untouched -- so one CUDA graph captured at
 * num_seqs requests and num_q_tokens tokens serves any smaller batch padded
 * with empty requests: q_len 0, context 0, seq_len 0, table row naming any
 * valid block; the padding tokens get slot -1 in pa_write_kv).
 * context_lens[b] tokens of it are already cached;
 * seq_lens[b] = context_lens[b] + q_len (int32 [num_seqs] each).  Its keys
 * 0..seq_lens[b]-1 live in the physical blocks block_tables[b][0..] (int32
 * [num_seqs][max_blocks_per_seq]; entries past ceil(seq_len/bs) are never
 * read).  New K/V must already be in the cache (pa_write_kv first, same
 * stream).  Query row i of request b (position context_lens[b] + i) attends
 * keys 0..context_lens[b]+i:
 *   out = softmax(scale * q k^T) v,  lse = ln sum_j exp(scale * q.k_j)
 * This one call covers decode rows (q_len 1), chunked-prefill chunks,
 * prefix-cache hits and speculative-verify rows (q_len 1 + k) in one batch.
 *   q      bf16 [num_q_tokens][num_q_heads][head_dim]
 *   out    bf16 [num_q_tokens][num_q_heads][head_dim]
 *   lse    fp32 [num_q_tokens][num_q_heads], or NULL
 * Rows with q_len * group <= 64 run on the split-KV memory-bound kernel;
 * longer requests run on the tcgen05 tensor-core kernel.
 */
int pa_attention(const void *q, const pa_kv_desc *kv, const int32_t *block_tables,
                 int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                 const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                 int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out, float *lse,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * One whole step in one call: pa_write_kv(k, v, slot_mapping,
 * num_new_tokens, kv) followed by pa_attention(q, kv, ...) on the same
 * stream, with the same arguments, rules, errors and results (caches bit for
 * bit, out and lse), in one host call: the same kernels run in the same
 * order, the write as a programmatic dependent of whatever ran before, so
 * its launch overlaps that kernel's tail and it is off the step's critical
 * path ([CH] §11.5: a decode step is dominated by fixed per-step costs;
 * this call halves the host calls per step).  num_seqs == 0 or
 * num_q_tokens == 0 does the write alone.
 */
int pa_write_kv_attention(const void *k, const void *v, const int64_t *slot_mapping,
                          int32_t num_new_tokens, const void *q, const pa_kv_desc *kv,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *query_start_loc, const int32_t *context_lens,
                          const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_tokens,
                          int32_t num_q_heads, float scale, void *out, float *lse,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_attention with the kernel choice exposed (tests, tuning):
 *   short_q_max_rows: a request whose q_len * group is at most this many
 *   rows runs on the split-KV kernel, the others on the tensor-core kernel.
 *   0 sends every request to the tensor-core kernel; -1 = default (64).
 *   Values above 64 are invalid.
 *   split_keys: 0 = automatic split-KV size; otherwise the number of keys per
 *   split (a multiple of 64) for the split-KV kernel.
 */
int pa_attention_ex(const void *q, const pa_kv_desc *kv, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                    const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                    int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out, float *lse,
                    void *workspace, size_t workspace_bytes, int32_t short_q_max_rows,
                    int32_t split_keys, void *stream);

/*
 * Merge operator of cascade inference ([AI] §02.1): combine two attention
 * states over disjoint key sets into the state over their union.
 *   M = max(lse_a, lse_b); lse = M + ln(e^(lse_a-M) + e^(lse_b-M))
 *   out = e^(lse_a-lse) o_a + e^(lse_b-lse) o_b
 * Two empty states (lse = -inf) give (0, -inf).  Associative and
 * commutative up to rounding.
 *   o_a, o_b, out        bf16 [n][num_heads][head_dim]
 *   lse_a, lse_b         fp32 [n][num_heads]
 *   lse_out              fp32 [n][num_heads], or NULL
 */
int pa_merge_states(const void *o_a, const float *lse_a, const void *o_b, const float *lse_b,
                    int32_t n, int32_t num_heads, int32_t head_dim, void *out, float *lse_out,
                    void *stream);

/*
 * pa_attention for callers that cannot allocate device memory (no
 * counterpart on the pages: this is a deployment convenience).  Same
 * arguments and results as pa_attention, without the workspace: the
 * library keeps its scratch (work list, split partial states, counters) in
 * one fixed device array of PA_NO_ALLOC_SCRATCH_BYTES.  The call allocates
 * nothing and frees nothing.
 *  - The array is committed on a device when this entry point is first
 *    called there (its module is loaded lazily; that first call also looks
 *    up the array's device address, with the device current) and is held
 *    until the process exits.  Make one call at start-up on each device you
 *    will use -- it may fail with PA_ERR_CUDA if the device is out of
 *    memory -- and before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents: calls whose kernels overlap on the GPU race and give wrong
 *    results.  Order them (one stream, or events).
 *  - A step whose work lists do not fit returns PA_ERR_WORKSPACE with a
 *    message.  The work lists get the least room that always fits, and the
 *    split-KV partial states what is left, so large batches may be cut into
 *    fewer, longer splits than pa_attention would choose (same results up
 *    to rounding).
 *  - On an fp8 (e4m3) pool there is no staging room for the tensor-core
 *    path: every request runs on the split-KV kernel (long ones in pieces of
 *    64 / group query tokens).
 */
#define PA_NO_ALLOC_SCRATCH_BYTES (32u << 20)
int pa_attention_no_alloc(const void *q, const pa_kv_desc *kv, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                          const int32_t *context_lens, const int32_t *seq_lens,
                          int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                          float scale, void *out, float *lse, void *stream);

/*
 * Workspace bytes for pa_prefix_attention / pa_cascade_decode.
 */
size_t pa_cascade_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t prefix_len);

/*
 * Extra workspace bytes, on top of pa_cascade_workspace_size, that
 * pa_prefix_attention and pa_cascade_decode need on an fp8 (e4m3) pool: the
 * prefix's ceil(prefix_len / block_size) blocks decoded to bf16 (exactly;
 * the per-kv-head scales are applied by the kernel) for the tensor-core
 * prefix pass, and their block list.  0 for an empty prefix; bf16 pools
 * need none.  A smaller workspace is refused with PA_ERR_WORKSPACE.
 * Returns 0 for invalid sizes.
 */
size_t pa_cascade_fp8_staging_bytes(int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t prefix_len);

/*
 * Shared-prefix ("multi-query") attention of cascade inference ([AI]
 * §02.1): every query row attends all prefix_len keys held, in order, by the
 * physical blocks prefix_blocks[0 .. ceil(prefix_len/bs)) (int32, device),
 * with no mask.  Each prefix block is loaded once per (kv head, 128 query
 * rows), not once per request; the key range is split over the SMs and the
 * splits' states are merged by a second launch within the call.  Writes
 * bf16 out and fp32 lse (may be NULL) shaped as in pa_attention.
 */
int pa_prefix_attention(const void *q, const pa_kv_desc *kv, const int32_t *prefix_blocks,
                        int32_t prefix_len, int32_t num_q_tokens, int32_t num_q_heads,
                        float scale, void *out, float *lse, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Cascade decode ([AI] §02.1) in one call: the shared-prefix pass above,
 * then paged attention over each request's unique suffix (block_tables,
 * context_lens and seq_lens describe the suffix alone: positions count from
 * the end of the prefix), with the prefix state folded into the suffix
 * pass's split-KV epilogue by the merge operator.  Equals pa_attention over
 * the full tables (prefix blocks followed by suffix blocks).
 */
int pa_cascade_decode(const void *q, const pa_kv_desc *kv, const int32_t *prefix_blocks,
                      int32_t prefix_len, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                      const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out,
                      float *lse, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Host-side check of step metadata (HOST pointers): qsl[0] == 0, qsl
 * non-decreasing and ending at or below num_q_tokens, seq_lens ==
 * context_lens + q_len,
 * every block id a request reads within [0, num_blocks), and (if
 * slot_mapping is not NULL) every slot either negative or inside the pool
 * and no slot used twice.  Returns PA_OK or PA_ERR_BAD_METADATA (with a
 * one-line reason in the thread-local buffer read by pa_last_error_message).
 */
int pa_validate_metadata(const int32_t *block_tables, int32_t max_blocks_per_seq,
                         const int32_t *query_start_loc, const int32_t *context_lens,
                         const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_tokens,
                         const int64_t *slot_mapping, int32_t num_blocks, int32_t block_size);

/* Reason for the last PA_ERR_* returned on this host thread ("" if none). */
const char *pa_last_error_message(void);

/* Static name of a return code. */
const char *pa_status_string(int code);

/*
 * Profiling hook.  After this call, every launch of kernel `which` made by
 * the calls above is bracketed by cudaEventRecord(start_event) and
 * cudaEventRecord(end_event) on the launch stream, so a caller can time one
 * kernel of a step with events.  While events are set for the split-KV or
 * the tensor-core kernel, pa_attention launches those two one after the
 * other (one tensor-core grid) instead of side by side; the results are
 * the same bit for bit.  Events are cudaEvent_t passed as void*; NULL
 * clears the hook.  The setting is process-wide; set it from one thread at
 * a time.
 *   which: PA_KERNEL_WRITE_KV, PA_KERNEL_PLAN, PA_KERNEL_SPLIT_KV,
 *          PA_KERNEL_TENSOR_CORE
 */
enum { PA_KERNEL_WRITE_KV = 0, PA_KERNEL_PLAN = 1, PA_KERNEL_SPLIT_KV = 2,
       PA_KERNEL_TENSOR_CORE = 3 };
int pa_set_profile_events(int32_t which, void *start_event, void *end_event);

/*
 * Test hook for the bounded device waits (no counterpart on the pages).
 * Every wait inside the kernels -- on a pipeline barrier, or the wait of a
 * step's last tensor-core grid for the CTAs of its first -- gives up after
 * 2 s, raises PA_DEV_WAIT_TIMEOUT, lets its copies in flight land and
 * returns; the context stays usable.  This hook makes one such wait run
 * out on purpose, so a test can check that path.  Nothing faults or traps.
 *   PA_TEST_STALL_NONE        normal operation (the default)
 *   PA_TEST_STALL_SPLIT_KV    in every later split-KV launch that waits for
 *                             its plan (not the mixed step's side-by-side
 *                             launch), CTA 0's producer stops after its
 *                             first stage: CTA 0's consumers wait for a
 *                             stage that never comes, time out and return.
 *                             The step's result is then incomplete.
 *   PA_TEST_STALL_LAST_GRID   in every later side-by-side step (split-KV
 *                             and tensor-core kernels together), the last
 *                             tensor-core grid waits for one CTA more than
 *                             the first grid launched.  All work is done
 *                             and the result is right; only the wait times
 *                             out.
 * Process-wide, read at launch time; set it from one thread, with no call
 * of this library in flight on the host.
 */
enum { PA_TEST_STALL_NONE = 0, PA_TEST_STALL_SPLIT_KV = 1, PA_TEST_STALL_LAST_GRID = 2 };
int pa_set_test_stall(int32_t which);

/*
 * Work counter of the tensor-core kernel (a check of its causal tile
 * skipping; "vLLM中如何实现大模型推理加速技术？", chunked prefill: a chunk's
 * score block covers only the keys up to its last row, 16^2*6 rather than
 * 16^2*9 for 48 tokens in 16-token tiles).  While `counter` (a DEVICE
 * pointer to one uint64) is set, every later launch of the tensor-core
 * kernel adds to it the number of 128-key tiles for which it issued Q K^T,
 * summed over its items (128-row query tile, kv head).  NULL (the default)
 * turns it off.  Process-wide; for tests, not for timed runs.
 */
int pa_set_tile_counter(uint64_t *counter);

/*
 * Read (and, if clear != 0, reset) the PA_DEV_* status word of the current
 * device.  Synchronises `stream` first.  HOST pointer `status`.
 */
int pa_read_device_status(uint32_t *status, int clear, void *stream);

/*
 * Number of kernels the library has enqueued in this process since it was
 * loaded, on any stream or device (launches recorded into a CUDA graph
 * count once, when captured; replays do not count).  Read it before and
 * after a region of calls to count their launches.  Thread-safe.
 */
uint64_t pa_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
