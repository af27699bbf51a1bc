// pa_shard.cpp -- request router for request-sharded replicas (declared in
// include/pa_shard.h).  Host-only.
//
// The data-parallel form of serving on the 2048ai.net page on the vLLM V1
// engine (data parallelism: a request router hands requests to full model
// replicas, and uneven load between replicas is the thing to avoid): each
// request of a step goes to one GPU, which runs its write and attention with
// no exchange.  Work is balanced on KV tokens read, by greedy longest-first
// list scheduling onto the least-loaded rank.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/pa.h"
#include "../../include/pa_shard.h"

extern "C" int pa_partition_requests(const int32_t *seq_lens, int32_t num_seqs,
                                     int32_t num_ranks, int32_t *rank_of_request,
                                     int64_t *rank_load) {
    if (num_seqs < 0 || num_ranks <= 0) return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_lens || !rank_of_request)) return PA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < num_seqs; ++b)
        if (seq_lens[b] < 0) return PA_ERR_INVALID_ARG;

    // heaviest first; equal weights keep request order
    std::vector<int32_t> order(static_cast<size_t>(num_seqs));
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return seq_lens[a] > seq_lens[b]; });

    // least-loaded rank on top; equal loads: the lowest rank
    using Entry = std::pair<int64_t, int32_t>;  // (load, rank)
    std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
    for (int32_t r = 0; r < num_ranks; ++r) heap.push({0, r});
    std::vector<int64_t> load(static_cast<size_t>(num_ranks), 0);
    for (const int32_t b : order) {
        const Entry top = heap.top();
        heap.pop();
        rank_of_request[b] = top.second;
        load[static_cast<size_t>(top.second)] = top.first + seq_lens[b];
        heap.push({top.first + seq_lens[b], top.second});
    }
    if (rank_load)
        for (int32_t r = 0; r < num_ranks; ++r) rank_load[r] = load[static_cast<size_t>(r)];
    return PA_OK;
}
