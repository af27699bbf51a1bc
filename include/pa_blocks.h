/*
 * pa_blocks.h -- host-side block manager of the paged KV pool, with a
 * content-hash prefix cache.  It is the step upstream of the attention path:
 * it decides which physical block holds each token of each request and emits
 * the block tables, slot mapping and lengths that pa_write_kv / pa_attention
 * consume.  Plain C ABI, host memory only; no CUDA call is made.
 *
 * Sources ("11. 推理加速(一):vLLM 原理", chuoer47.github.io):
 *  §11.2 PagedAttention: the KV cache is cut into fixed-size blocks; each
 *        request keeps a block table (logical block -> physical block); the
 *        physical blocks need not be contiguous; a new physical block is
 *        allocated only when the request's tokens reach it; two requests with
 *        the same prefix point their tables at the same physical blocks
 *        (block tables [3,7,11] and [3,7,5]), and a shared block that would
 *        be written gets a copy first (copy-on-write).
 *  §11.4 Prefix caching: every full block is identified by a hash of its
 *        token ids; a new request first looks for cached blocks with its
 *        hashes and references them (ref_count++) instead of computing them
 *        again, so only the tokens after the hit are prefilled.
 *
 * Readings where the page is silent:
 *  - A block's identity is its whole token prefix (tokens 0 .. end of the
 *    block), hashed as a 128-bit chain block by block: a token's K/V depends
 *    on every token before it, so equal block contents under different
 *    prefixes are different blocks.  Only full blocks are cached.
 *  - Prefix matching runs from block 0 and stops at the first miss.  At
 *    least the prompt's last token is always computed (a prompt whose every
 *    block is cached keeps its last block out of the hit).
 *  - Allocation takes the lowest-numbered free block; when none is free it
 *    evicts the cached, unreferenced block released longest ago (blocks of a
 *    finished request are released from its last block to its first).  A
 *    newly filled block whose prefix is already cached in another block
 *    stays uncached.
 *  - Copy-on-write: before a request writes into a partially filled block
 *    that other requests also reference (after pa_bm_fork), the block is
 *    replaced in its table by a fresh copy; the copy (src -> dst physical
 *    block) is reported to the caller, who copies the K/V bytes.
 *
 * Errors: every call returns PA_OK (0) or a PA_ERR_* code (pa.h); on an
 * error nothing changes.  PA_ERR_WORKSPACE here means "not enough free
 * blocks" (the caller's scheduler would preempt or wait).
 */
#ifndef PA_BLOCKS_H_
#define PA_BLOCKS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

/* A manager of num_blocks physical blocks of block_size tokens (> 0 each).
 * Returns NULL on invalid sizes or out of host memory. */
pa_block_manager *pa_bm_create(int32_t num_blocks, int32_t block_size);
void pa_bm_destroy(pa_block_manager *bm);

/* Admit request req_id (not yet present) with its prompt token ids
 * (num_tokens >= 1).  Matches cached full blocks of the prompt's prefix and
 * references them; *num_cached_tokens (optional) receives the number of
 * prompt tokens whose K/V is already cached (a multiple of block_size).  No
 * block is allocated here. */
int pa_bm_add_request(pa_block_manager *bm, int64_t req_id, const int32_t *token_ids,
                      int32_t num_tokens, int32_t *num_cached_tokens);

/* Append token ids (e.g. sampled tokens) to a request's sequence. */
int pa_bm_append_tokens(pa_block_manager *bm, int64_t req_id, const int32_t *token_ids,
                        int32_t num_tokens);

/* New request dst_id sharing everything of src_id (tokens, computed tokens,
 * every block, each block's reference count + 1). */
int pa_bm_fork(pa_block_manager *bm, int64_t src_id, int64_t dst_id);

/*
 * One step: request req_ids[i] computes its next num_new_tokens[i] (>= 1)
 * tokens, which must already be in its sequence.  Allocates the blocks the
 * new tokens need (copy-on-write first where needed), writes the step's
 * metadata in the layout pa_attention takes, marks the tokens computed and
 * caches every block they fill.  Outputs (caller-allocated host arrays):
 *   block_tables     int32 [num_reqs][max_blocks_per_seq], -1 past each table
 *   query_start_loc  int32 [num_reqs + 1]
 *   context_lens     int32 [num_reqs]  (tokens computed before the step)
 *   seq_lens         int32 [num_reqs]
 *   slot_mapping     int64 [sum of num_new_tokens]
 *   copies           int32 [max_copies][2] (src, dst) physical blocks to copy
 *                    before the step's write; *num_copies receives the count
 * PA_ERR_INVALID_ARG: unknown or repeated request, a token not yet appended,
 * a table wider than max_blocks_per_seq, or more copies than max_copies.
 * PA_ERR_WORKSPACE: not enough free + evictable blocks.
 */
int pa_bm_schedule(pa_block_manager *bm, int32_t num_reqs, const int64_t *req_ids,
                   const int32_t *num_new_tokens, int32_t max_blocks_per_seq,
                   int32_t *block_tables, int32_t *query_start_loc, int32_t *context_lens,
                   int32_t *seq_lens, int64_t *slot_mapping, int32_t max_copies,
                   int32_t *copies, int32_t *num_copies);

/* Finish a request: its blocks are released (last block first); cached
 * blocks stay matchable until evicted, others become free. */
int pa_bm_free_request(pa_block_manager *bm, int64_t req_id);

/* Introspection (tests, schedulers). */
int32_t pa_bm_num_free_blocks(const pa_block_manager *bm);      /* free + evictable */
int32_t pa_bm_num_cached_blocks(const pa_block_manager *bm);    /* blocks matchable by hash */
int32_t pa_bm_block_ref_count(const pa_block_manager *bm, int32_t block);  /* -1: bad id */
/* Copies request req_id's block table into out (capacity cap); returns its
 * length, or -1 for an unknown request. */
int32_t pa_bm_request_blocks(const pa_block_manager *bm, int64_t req_id, int32_t *out,
                             int32_t cap);
/* Tokens of req_id whose K/V is computed, or -1 for an unknown request. */
int32_t pa_bm_num_computed(const pa_block_manager *bm, int64_t req_id);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCKS_H_ */
