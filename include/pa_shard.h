/*
 * pa_shard.h -- C ABI of libpa's request router for request-sharded replicas.
 *
 * Source: 2048ai.net page on the vLLM V1 engine, section on data parallelism:
 * every device holds a full replica, a request router hands each request to
 * one device, each device runs its requests end to end with no exchange in
 * the middle, and the main weakness is load imbalance between replicas.  For
 * the paged-attention step the work of a request is dominated by the KV it
 * reads (every visible K/V row once per kv head), so the router balances KV
 * tokens: greedy longest-first assignment to the least-loaded rank.
 *
 * Host-only: every pointer is a HOST pointer; nothing touches a GPU.  The
 * result is deterministic (ties broken by request index, then by rank).
 */
#ifndef PA_SHARD_H_
#define PA_SHARD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Assign num_seqs requests to num_ranks replicas.  Request b weighs
 * seq_lens[b] KV tokens (its K/V bytes are that times 2 * num_kv_heads *
 * head_dim * element size, the same factor for every request).  Requests are
 * taken heaviest first (equal weights in request order) and each goes to the
 * rank with the least weight so far (equal loads: the lowest rank).  So the
 * heaviest and the lightest rank differ by at most one request's weight.
 *   seq_lens         int32 [num_seqs], each >= 0
 *   rank_of_request  int32 [num_seqs] out: the rank of each request
 *   rank_load        int64 [num_ranks] out (may be NULL): KV tokens per rank
 * Returns PA_OK (0), or PA_ERR_INVALID_ARG (1) for num_seqs < 0,
 * num_ranks <= 0, a NULL array or a negative length (outputs untouched).
 */
int pa_partition_requests(const int32_t *seq_lens, int32_t num_seqs, int32_t num_ranks,
                          int32_t *rank_of_request, int64_t *rank_load);

#ifdef __cplusplus
}
#endif
#endif /* PA_SHARD_H_ */
