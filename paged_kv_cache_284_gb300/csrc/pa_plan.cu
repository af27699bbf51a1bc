// pa_plan.cu -- device-side step planner.
//
// From the step's AttentionMeta-style metadata (query_start_loc,
// context_lens, seq_lens; "vLLM中如何实现大模型推理加速技术？": every attention
// op carries each request's progress) it classifies each request, picks a
// split-KV size and writes the two work lists into the workspace:
//   * short rows (q_len * group <= short_max_rows: decode, speculative
//     verify, small chunks) -> split-KV items (request, kv head, key range);
//   * long rows (chunked-prefill chunks, prefix-hit prompts, whole prompts)
//     -> tensor-core items (request, kv head, 128-row query tile).
// Runs as one CTA so the whole step stays on the device (no host round trip,
// capturable in a CUDA graph).  It also zeroes the split completion
// counters and the dynamic work counters.
#include "pa_internal.cuh"

namespace pa {

// Exclusive block-wide prefix sum over kPlanThreads threads.
__device__ int block_exclusive_scan(int v, int *tmp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (kPlanThreads / 32)) ? tmp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        tmp[lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == 31) tmp[32] = wi;
    }
    __syncthreads();
    const int res = tmp[warp] + incl - v;
    *total = tmp[32];
    __syncthreads();
    return res;
}

__device__ long long block_sum_ll(long long v, long long *tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        long long w = (lane < (kPlanThreads / 32)) ? tmp[lane] : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (lane == 0) tmp[32] = w;
    }
    __syncthreads();
    const long long r = tmp[32];
    __syncthreads();
    return r;
}

struct ReqInfo {
    int n, ctx, len;
    int is_short;
    int pieces;   // query pieces of a split-KV request
    int qtiles;   // query tiles of a tensor-core request
};

__device__ __forceinline__ ReqInfo load_req(const PlanParams &p, int b) {
    ReqInfo r{};
    const int q0 = p.qsl[b], q1 = p.qsl[b + 1];
    r.n = q1 - q0;
    r.ctx = p.ctx[b];
    r.len = p.seq_lens[b];
    const bool bad = r.n < 0 || r.ctx < 0 || r.len != r.ctx + r.n || q0 < 0 ||
                     q1 > p.num_q_tokens;
    if (bad) {
        flag_status(p.status, PA_DEV_BAD_METADATA);
        r.n = 0;
    }
    if (r.n > 0) {
        r.is_short = (static_cast<long long>(r.n) * p.group <= p.short_max_rows) ? 1 : 0;
        // fp8 pool: a long request without a staging copy runs as pieces
        if (p.fp8 && !r.is_short && !(p.stage_cap > 0 && p.stage_base[b] >= 0)) r.is_short = 1;
        if (r.is_short)
            r.pieces = (r.n + p.piece_tokens - 1) / p.piece_tokens;
        else
            r.qtiles = (r.n + p.q_tile_tokens - 1) / p.q_tile_tokens;
    }
    return r;
}

// Piece i of a split-KV request: its query tokens and the 64-key stages up
// to its last token's causal limit.
struct Piece {
    int q_begin, q_count, stages;
};
__device__ __forceinline__ Piece piece_of(const PlanParams &p, const ReqInfo &r, int i) {
    Piece pc;
    pc.q_begin = i * p.piece_tokens;
    pc.q_count = min(p.piece_tokens, r.n - pc.q_begin);
    pc.stages = (r.ctx + pc.q_begin + pc.q_count + kStageKeys - 1) / kStageKeys;
    return pc;
}

constexpr int kSortBins = kPlanThreads;  // bins of the longest-first sort

// Sort bin of query tile qt of a long request: bin 0 holds the most 128-key
// tiles.
__device__ __forceinline__ int long_bin(const PlanParams &p, const ReqInfo &r, int qt) {
    const int nvalid = min(p.q_tile_tokens, r.n - qt * p.q_tile_tokens);
    const int kend = min(r.len, r.ctx + qt * p.q_tile_tokens + nvalid);
    const int tiles = (kend + kLongKeys - 1) / kLongKeys;
    return kSortBins - 1 - min(tiles, kSortBins - 1);
}

// Sort bin of a split-KV item of `stages` stages: bin 0 holds the longest.
__device__ __forceinline__ int short_bin(int stages) {
    return kSortBins - 1 - min(stages, kSortBins - 1);
}

// First stage of split s of ns over `stages` stages (s = ns gives the end).
__device__ __forceinline__ int split_begin(int stages, int ns, int s) {
    return static_cast<int>(static_cast<long long>(stages) * s / ns);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
    __shared__ int tmp[33];
    __shared__ long long tmpl[33];
    __shared__ int bins[kSortBins];
    __shared__ int s_split, s_overflow, s_max_stages;
    const int tid = threadIdx.x, lane = tid & 31;
    const int hkv = p.num_kv_heads;
    // the metadata (and the workspace) may belong to the previous kernel
    pdl_wait();
    pdl_trigger();
    if (tid == 0) {
        s_overflow = 0;
        s_max_stages = 0;
    }
    for (int i = tid; i < kSortBins; i += kPlanThreads) bins[i] = 0;
    // 0. fp8 pool with a staging area: long requests get consecutive bf16
    // staging blocks in request order while they fit (a request that does
    // not fit, and every later one, runs as split-KV pieces instead).
    int staged = 0, staged_blocks = 0;
    if (p.fp8 && p.stage_cap > 0) {
        int cand_base = 0;
        for (int b0 = 0; b0 < p.num_seqs; b0 += kPlanThreads) {
            const int b = b0 + tid;
            int cnt = 0;
            if (b < p.num_seqs) {
                const int n = p.qsl[b + 1] - p.qsl[b], len = p.seq_lens[b];
                if (n > 0 && len > 0 && static_cast<long long>(n) * p.group > p.short_max_rows)
                    cnt = (len + p.block_size - 1) / p.block_size;
            }
            int tot_c, tot_s;
            const int base = cand_base + block_exclusive_scan(cnt, tmp, &tot_c);
            const bool fits = cnt > 0 && base + cnt <= p.stage_cap;
            const int idx = staged + block_exclusive_scan(fits ? 1 : 0, tmp, &tot_s);
            if (b < p.num_seqs) p.stage_base[b] = fits ? base : -1;
            if (fits) p.stage_list[idx] = b;
            staged_blocks += static_cast<int>(block_sum_ll(fits ? cnt : 0, tmpl));
            cand_base += tot_c;
            staged += tot_s;
        }
        __syncthreads();
    }
    // Request tid's metadata is read once and kept in registers; only steps
    // with more than kPlanThreads requests read the others again per pass.
    const ReqInfo mine = tid < p.num_seqs ? load_req(p, tid) : ReqInfo{};
    auto req = [&](int b) { return b == tid ? mine : load_req(p, b); };
    __syncthreads();

    // 1. total split-KV work (in stages) -------------------------------------
    long long work = 0;
    int max_stages = 0, pieces = 0;
    for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
        const ReqInfo r = req(b);
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            work += pc.stages;
            max_stages = max(max_stages, pc.stages);
        }
        pieces += r.pieces;
    }
    max_stages = __reduce_max_sync(0xffffffffu, max_stages);
    if (lane == 0 && max_stages > 0) atomicMax(&s_max_stages, max_stages);
    const long long total_work = block_sum_ll(work, tmpl) * hkv;  // also orders the atomics
    const long long total_pieces = block_sum_ll(pieces, tmpl);

    // 2. split size ------------------------------------------------------------
    int sp;
    if (p.split_stages > 0) {
        sp = p.split_stages;
    } else {
        const long long tgt = max(1, p.target_items);
        sp = static_cast<int>(max(static_cast<long long>(kMinSplitStages),
                                  (total_work + tgt - 1) / tgt));
    }
    for (int guard = 0; guard < 40; ++guard) {
        long long items = 0, rows = 0;
        for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
            const ReqInfo r = req(b);
            for (int i = 0; i < r.pieces; ++i) {
                const Piece pc = piece_of(p, r, i);
                const int ns = (pc.stages + sp - 1) / sp;
                items += ns;
                if (ns > 1) rows += static_cast<long long>(ns) * pc.q_count * p.group;
            }
        }
        items = block_sum_ll(items, tmpl) * hkv;
        rows = block_sum_ll(rows, tmpl) * hkv;
        if ((items <= p.max_short && rows <= p.cap_rows) || sp >= s_max_stages) break;
        sp *= 2;
    }
    if (tid == 0) {
        s_split = sp;
        if (total_pieces * hkv > p.num_counters) s_overflow = 1;
    }
    __syncthreads();
    sp = s_split;

    int short_base = 0, long_base = 0, row_base = 0, piece_base = 0;

    // 3. split-KV items, longest key range first (counting sort on the number
    // of stages of the item).  A piece's ns splits cut its stages into ranges
    // that differ by at most one stage.  Partial-state rows and completion
    // counters are handed out in request order by block scans.
    for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
        const ReqInfo r = req(b);
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            const int ns = (pc.stages + sp - 1) / sp;
            for (int s = 0; s < ns; ++s)
                atomicAdd(&bins[short_bin(split_begin(pc.stages, ns, s + 1) -
                                          split_begin(pc.stages, ns, s))],
                          1);
        }
    }
    __syncthreads();
    {
        int tot_s;
        const int v = tid < kSortBins ? bins[tid] : 0;
        const int off = block_exclusive_scan(v, tmp, &tot_s);
        if (tid < kSortBins) bins[tid] = off;
        short_base = tot_s;  // records
        __syncthreads();
    }
    for (int b0 = 0; b0 < p.num_seqs; b0 += kPlanThreads) {
        const int b = b0 + tid;
        ReqInfo r{};
        if (b < p.num_seqs) r = req(b);
        int n_rows = 0;
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            const int ns = (pc.stages + sp - 1) / sp;
            if (ns > 1) n_rows += ns * pc.q_count * p.group * hkv;
        }
        int tot_r, tot_p;
        const int off_r = row_base + block_exclusive_scan(n_rows, tmp, &tot_r);
        const int off_p = piece_base + block_exclusive_scan(r.pieces, tmp, &tot_p);
        row_base += tot_r;
        piece_base += tot_p;
        if (static_cast<long long>(short_base) * hkv > p.max_short || row_base > p.cap_rows ||
            s_overflow) {
            if (tid == 0) s_overflow = 1;
            continue;  // uniform: the totals are block-wide and s_overflow was set before a barrier
        }
        int row = off_r;
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            const int ns = (pc.stages + sp - 1) / sp;
            const int R = pc.q_count * p.group;
            for (int s = 0; s < ns; ++s) {
                const int s0 = split_begin(pc.stages, ns, s);
                const int s1 = split_begin(pc.stages, ns, s + 1);
                ShortItem it;
                it.b = b;
                it.split = s;
                it.nsplit = ns;
                it.stage_begin = s0;
                it.stage_end = s1;
                it.partial_base = (ns > 1) ? row + s * R : 0;
                it.q_begin = pc.q_begin;
                it.q_count = pc.q_count;
                it.counter = off_p + i;
                it.pad0 = it.pad1 = it.pad2 = 0;
                store_record(p.short_items, atomicAdd(&bins[short_bin(s1 - s0)], 1), it);
            }
            if (ns > 1) row += ns * R * hkv;
        }
    }
    __syncthreads();

    // 3b. tensor-core items, longest key range first (counting sort on the
    // number of 128-key tiles), so persistent CTAs that take items in order
    // finish together.
    for (int i = tid; i < kSortBins; i += kPlanThreads) bins[i] = 0;
    __syncthreads();
    for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
        const ReqInfo r = req(b);
        for (int qt = 0; qt < r.qtiles; ++qt)
            atomicAdd(&bins[long_bin(p, r, qt)], 1);
    }
    __syncthreads();
    {
        // one bin per thread: exclusive scan gives each bin's first slot
        int tot_l;
        const int v = tid < kSortBins ? bins[tid] : 0;
        const int off = block_exclusive_scan(v, tmp, &tot_l);
        if (tid < kSortBins) bins[tid] = off;
        long_base = tot_l;
        __syncthreads();
    }
    if (static_cast<long long>(long_base) * hkv > p.max_long) {
        if (tid == 0) s_overflow = 1;
    } else {
        for (int b = tid; b < p.num_seqs; b += kPlanThreads) {
            const ReqInfo r = req(b);
            for (int qt = 0; qt < r.qtiles; ++qt) {
                const int nvalid = min(p.q_tile_tokens, r.n - qt * p.q_tile_tokens);
                LongItem it{};
                it.b = b;
                it.q_tile = qt;
                it.key_begin = 0;
                it.key_end = min(r.len, r.ctx + qt * p.q_tile_tokens + nvalid);
                store_record(p.long_items, atomicAdd(&bins[long_bin(p, r, qt)], 1), it);
            }
        }
    }

    // 4. counters and header ----------------------------------------------------
    for (int i = tid; i < p.num_counters; i += kPlanThreads) p.counters[i] = 0;
    __syncthreads();
    if (tid == 0) {
        // A work list that did not fit is never run partially: no items at all.
        if (s_overflow) flag_status(p.status, PA_DEV_PLAN_OVERFLOW);
        p.hdr->num_short_items = s_overflow ? 0 : short_base * hkv;
        p.hdr->num_long_items = s_overflow ? 0 : long_base * hkv;
        p.hdr->short_next = 0;
        p.hdr->long_next = 0;
        p.hdr->split_stages = sp;
        p.hdr->partial_rows = row_base;
        p.hdr->num_staged = s_overflow ? 0 : staged;
        p.hdr->first_done = 0;
        p.hdr->staged_blocks = s_overflow ? 0 : staged_blocks;
    }
}

int launch_plan(const PlanParams &p, cudaStream_t s) {
    PdlLaunch l(1, kPlanThreads, 0, s);
    return cudaLaunchKernelEx(&l.cfg, plan_kernel, p) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
