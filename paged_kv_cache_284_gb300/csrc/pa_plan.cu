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

// Exclusive block-wide prefix sum over the kT threads of the block.
template <int kT>
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
        int w = (lane < (kT / 32)) ? tmp[lane] : 0;
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

// Exact warp sum of non-negative 64-bit values with single-instruction warp
// reductions: three slices of 21, 21 and 22 bits are summed separately (32
// lanes x 2^22 < 2^32, so no slice overflows) and recombined.
__device__ __forceinline__ long long warp_sum_ll(long long x) {
    const unsigned long long v = static_cast<unsigned long long>(x);
    const unsigned a = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v & 0x1fffffu));
    const unsigned b = __reduce_add_sync(0xffffffffu, static_cast<unsigned>((v >> 21) & 0x1fffffu));
    const unsigned c = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v >> 42));
    return static_cast<long long>(a + (static_cast<unsigned long long>(b) << 21) +
                                  (static_cast<unsigned long long>(c) << 42));
}

// Block-wide sums of N non-negative 64-bit values and the maximum of one
// non-negative int, all in one pass (two barriers for the lot).
constexpr int kRedStride = kPlanThreads / 32 + 1;
template <int kT, int N>
__device__ void block_reduce(long long (&v)[N], int &mx, long long *tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = warp_sum_ll(v[i]);
    mx = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(mx)));
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < N; ++i) tmp[i * kRedStride + warp] = v[i];
        tmp[N * kRedStride + warp] = mx;
    }
    __syncthreads();
    if (warp == 0) {
        const bool in = lane < kT / 32;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const long long w = warp_sum_ll(in ? tmp[i * kRedStride + lane] : 0);
            if (lane == 0) tmp[i * kRedStride + 32] = w;
        }
        const unsigned m = __reduce_max_sync(
            0xffffffffu, in ? static_cast<unsigned>(tmp[N * kRedStride + lane]) : 0u);
        if (lane == 0) tmp[N * kRedStride + 32] = m;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = tmp[i * kRedStride + 32];
    mx = static_cast<int>(tmp[N * kRedStride + 32]);
    __syncthreads();
}

// Exclusive block-wide prefix sums of two values at once (tmp: 66 ints).
template <int kT>
__device__ void block_exclusive_scan2(int a, int b, int *tmp, int &pa, int &pb, int &ta, int &tb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int na = __shfl_up_sync(0xffffffffu, ia, o);
        const int nb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += na;
            ib += nb;
        }
    }
    if (lane == 31) {
        tmp[warp] = ia;
        tmp[33 + warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        const bool in = lane < kT / 32;
        const int wa = in ? tmp[lane] : 0, wb = in ? tmp[33 + lane] : 0;
        int sa = wa, sb = wb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int na = __shfl_up_sync(0xffffffffu, sa, o);
            const int nb = __shfl_up_sync(0xffffffffu, sb, o);
            if (lane >= o) {
                sa += na;
                sb += nb;
            }
        }
        tmp[lane] = sa - wa;
        tmp[33 + lane] = sb - wb;
        if (lane == 31) {
            tmp[32] = sa;
            tmp[65] = sb;
        }
    }
    __syncthreads();
    pa = tmp[warp] + ia - a;
    pb = tmp[33 + warp] + ib - b;
    ta = tmp[32];
    tb = tmp[65];
    __syncthreads();
}

template <int kT>
__device__ long long block_sum_ll(long long v, long long *tmp) {
    long long a[1] = {v};
    int m = 0;
    block_reduce<kT, 1>(a, m, tmp);
    return a[0];
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

// The longest-first sorts are counting sorts with one bin per thread (kT
// bins); a bin holds 2^shift consecutive lengths, the least shift that fits
// the step's longest item, so a small plan still sorts long items closely.
__device__ __forceinline__ int bin_shift(int longest, int bins) {
    int sh = 0;
    while ((longest >> sh) >= bins) ++sh;
    return sh;
}

// 128-key tiles of query tile qt of a long request.
__device__ __forceinline__ int long_tiles(const PlanParams &p, const ReqInfo &r, int qt) {
    const int nvalid = min(p.q_tile_tokens, r.n - qt * p.q_tile_tokens);
    const int kend = min(r.len, r.ctx + qt * p.q_tile_tokens + nvalid);
    return (kend + kLongKeys - 1) / kLongKeys;
}

// Sort bin of an item of `len` stages (or tiles): bin 0 holds the longest.
__device__ __forceinline__ int len_bin(int len, int shift, int bins) {
    return bins - 1 - min(len >> shift, bins - 1);
}

// A piece of `stages` stages cut into ns splits whose ranges differ by at
// most one stage: the first `rem` splits take q + 1 stages, the others q.
struct SplitCut {
    int ns, q, rem;
};
__device__ __forceinline__ SplitCut split_cut(int stages, int sp) {
    SplitCut c;
    c.ns = (stages + sp - 1) / sp;
    c.q = stages / c.ns;
    c.rem = stages - c.q * c.ns;
    return c;
}

// kT threads: 1024 in general, one warp for steps of few requests (its
// phases then cost shuffles instead of block barriers).
template <int kT>
__global__ void __launch_bounds__(kT) plan_kernel(PlanParams p) {
    constexpr int kSortBins = kT;
    __shared__ int tmp[66];
    __shared__ long long tmpl[5 * kRedStride];
    __shared__ int bins[kSortBins];
    __shared__ int s_overflow;
    const int tid = threadIdx.x;
    const int hkv = p.num_kv_heads;
    // the metadata (and the workspace) may belong to the previous kernel
    pdl_wait();
    pdl_trigger();
    if (tid == 0) s_overflow = 0;
    for (int i = tid; i < kSortBins; i += kT) bins[i] = 0;
    // 0. fp8 pool with a staging area: long requests get consecutive bf16
    // staging blocks in request order while they fit (a request that does
    // not fit, and every later one, runs as split-KV pieces instead).
    int staged = 0, staged_blocks = 0;
    if (p.fp8 && p.stage_cap > 0) {
        int cand_base = 0;
        for (int b0 = 0; b0 < p.num_seqs; b0 += kT) {
            const int b = b0 + tid;
            int cnt = 0;
            if (b < p.num_seqs) {
                const int n = p.qsl[b + 1] - p.qsl[b], len = p.seq_lens[b];
                if (n > 0 && len > 0 && static_cast<long long>(n) * p.group > p.short_max_rows)
                    cnt = (len + p.block_size - 1) / p.block_size;
            }
            int tot_c, tot_s;
            const int base = cand_base + block_exclusive_scan<kT>(cnt, tmp, &tot_c);
            const bool fits = cnt > 0 && base + cnt <= p.stage_cap;
            const int idx = staged + block_exclusive_scan<kT>(fits ? 1 : 0, tmp, &tot_s);
            if (b < p.num_seqs) p.stage_base[b] = fits ? base : -1;
            if (fits) p.stage_list[idx] = b;
            staged_blocks += static_cast<int>(block_sum_ll<kT>(fits ? cnt : 0, tmpl));
            cand_base += tot_c;
            staged += tot_s;
        }
        __syncthreads();
    }
    // Request tid's metadata is read once and kept in registers; only steps
    // with more than kT requests read the others again per pass.
    const ReqInfo mine = tid < p.num_seqs ? load_req(p, tid) : ReqInfo{};
    auto req = [&](int b) { return b == tid ? mine : load_req(p, b); };
    __syncthreads();

    // 1. totals: split-KV work (in stages), pieces, longest piece, query tiles
    long long tot[3] = {0, 0, 0};  // work, pieces, tensor-core query tiles
    int max_stages = 0;
    for (int b = tid; b < p.num_seqs; b += kT) {
        const ReqInfo r = req(b);
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            tot[0] += pc.stages;
            max_stages = max(max_stages, pc.stages);
        }
        tot[1] += r.pieces;
        tot[2] += r.qtiles;
    }
    block_reduce<kT, 3>(tot, max_stages, tmpl);
    const long long total_work = tot[0] * hkv;
    const long long total_pieces = tot[1];
    const long long total_qtiles = tot[2];

    // 2. split size ------------------------------------------------------------
    // A split-KV item costs its stages plus a fixed cost (first-data latency
    // and the split epilogue) worth a few stages.  When every piece can have
    // a CTA of its own (P <= C items unsplit), the cut aims at one item per
    // CTA, so that all items run in a single round: sum_i ceil(s_i / sp) <=
    // W / sp + P, so sp = W / (C - P) always fits, and W / (C - P / 2) (half
    // an item of rounding per piece) usually does and gives shorter items.
    // Otherwise items aim at about target_items, so that longest-first
    // dynamic scheduling balances the CTAs (see below).  One counting pass checks both
    // candidates and the work-list capacities; the doubling loop below runs
    // only if they overflow.  (32-bit arithmetic: W saturates, which only
    // coarsens the heuristic.)
    const int W = static_cast<int>(min(total_work, 1LL << 30));
    const int P = static_cast<int>(min(total_pieces * hkv, 1LL << 30));
    const int C = max(1, p.num_ctas);
    int sp_a = kMinSplitStages, sp_b = kMinSplitStages;
    if (p.split_stages > 0) {
        sp_a = sp_b = p.split_stages;
    } else if (W > 0 && P <= C) {
        const int da = C - P / 2;
        sp_a = max(kMinSplitStages, (W + da - 1) / da);
        sp_b = P < C ? max(kMinSplitStages, (W + (C - P) - 1) / (C - P)) : max(sp_a, max_stages);
    } else if (W > 0) {
        // about target_items items, but no smaller than a cut into k =
        // ceil(P / C) rounds needs (kC - P/2 > 0), capped at 3/4 of the
        // average per-CTA load so that the longest items still balance;
        // measured 3 % faster than target_items alone on decode batches of
        // 40-64 requests and on the cascade suffix, even elsewhere
        const int tgt = max(1, p.target_items);
        const int sp_t = max(kMinSplitStages, (W + tgt - 1) / tgt);
        const long long kC = static_cast<long long>((P + C - 1) / C) * C;
        const int da = static_cast<int>(kC - P / 2);
        const int sp_k = max(kMinSplitStages, (W + da - 1) / da);
        const int cap = static_cast<int>(3LL * W / (4LL * C));
        sp_a = sp_b = max(sp_t, min(sp_k, cap));
    }
    long long cnt[4] = {0, 0, 0, 0};  // items and partial-state rows at sp_a, at sp_b
    for (int b = tid; b < p.num_seqs; b += kT) {
        const ReqInfo r = req(b);
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            const int na = (pc.stages + sp_a - 1) / sp_a, nb = (pc.stages + sp_b - 1) / sp_b;
            cnt[0] += na;
            cnt[2] += nb;
            if (na > 1) cnt[1] += static_cast<long long>(na) * pc.q_count * p.group;
            if (nb > 1) cnt[3] += static_cast<long long>(nb) * pc.q_count * p.group;
        }
    }
    {
        int unused = 0;
        block_reduce<kT, 4>(cnt, unused, tmpl);
    }
    const bool one_round = p.split_stages <= 0 && W > 0 && P <= C;
    const bool use_a = !one_round || cnt[0] * hkv <= C;
    int sp = use_a ? sp_a : sp_b;
    long long items = (use_a ? cnt[0] : cnt[2]) * hkv, rows = (use_a ? cnt[1] : cnt[3]) * hkv;
    for (int guard = 0; guard < 40; ++guard) {
        if ((items <= p.max_short && rows <= p.cap_rows) || sp >= max_stages) break;
        sp *= 2;
        long long c2[2] = {0, 0};
        for (int b = tid; b < p.num_seqs; b += kT) {
            const ReqInfo r = req(b);
            for (int i = 0; i < r.pieces; ++i) {
                const Piece pc = piece_of(p, r, i);
                const int ns = (pc.stages + sp - 1) / sp;
                c2[0] += ns;
                if (ns > 1) c2[1] += static_cast<long long>(ns) * pc.q_count * p.group;
            }
        }
        int unused = 0;
        block_reduce<kT, 2>(c2, unused, tmpl);
        items = c2[0] * hkv;
        rows = c2[1] * hkv;
    }
    if (tid == 0 && total_pieces * hkv > p.num_counters) s_overflow = 1;
    // no split-KV item is longer than sp stages or than the longest piece
    const int shift_s = bin_shift(min(sp, max_stages), kSortBins);

    int short_base = 0, long_base = 0, row_base = 0, piece_base = 0;

    // 3. split-KV items, longest key range first (counting sort on the number
    // of stages of the item).  A piece's splits of equal length take
    // consecutive slots of their bin, reserved with one atomic.  Partial-state
    // rows and completion counters are handed out in request order by block
    // scans.
    for (int b = tid; b < p.num_seqs; b += kT) {
        const ReqInfo r = req(b);
        for (int i = 0; i < r.pieces; ++i) {
            const SplitCut c = split_cut(piece_of(p, r, i).stages, sp);
            if (c.rem > 0) atomicAdd(&bins[len_bin(c.q + 1, shift_s, kSortBins)], c.rem);
            if (c.ns > c.rem) atomicAdd(&bins[len_bin(c.q, shift_s, kSortBins)], c.ns - c.rem);
        }
    }
    __syncthreads();
    {
        int tot_s;
        const int v = tid < kSortBins ? bins[tid] : 0;
        const int off = block_exclusive_scan<kT>(v, tmp, &tot_s);
        if (tid < kSortBins) bins[tid] = off;
        short_base = tot_s;  // records
        __syncthreads();
    }
    for (int b0 = 0; b0 < p.num_seqs; b0 += kT) {
        const int b = b0 + tid;
        ReqInfo r{};
        if (b < p.num_seqs) r = req(b);
        int n_rows = 0;
        for (int i = 0; i < r.pieces; ++i) {
            const Piece pc = piece_of(p, r, i);
            const int ns = (pc.stages + sp - 1) / sp;
            if (ns > 1) n_rows += ns * pc.q_count * p.group * hkv;
        }
        int off_r, off_p, tot_r, tot_p;
        block_exclusive_scan2<kT>(n_rows, r.pieces, tmp, off_r, off_p, tot_r, tot_p);
        off_r += row_base;
        off_p += piece_base;
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
            const SplitCut c = split_cut(pc.stages, sp);
            const int R = pc.q_count * p.group;
            const int slot_hi =
                c.rem > 0 ? atomicAdd(&bins[len_bin(c.q + 1, shift_s, kSortBins)], c.rem) : 0;
            const int slot_lo =
                c.ns > c.rem ? atomicAdd(&bins[len_bin(c.q, shift_s, kSortBins)], c.ns - c.rem)
                             : 0;
            ShortItem it;
            it.b = b;
            it.nsplit = c.ns;
            it.q_begin = pc.q_begin;
            it.q_count = pc.q_count;
            it.counter = off_p + i;
            it.seq_len = r.len;
            it.pad1 = it.pad2 = 0;
            for (int s = 0; s < c.ns; ++s) {
                const bool big = s < c.rem;
                it.split = s;
                it.stage_begin = s * c.q + min(s, c.rem);
                it.stage_end = it.stage_begin + c.q + (big ? 1 : 0);
                it.partial_base = (c.ns > 1) ? row + s * R : 0;
                store_record(p.short_items, big ? slot_hi + s : slot_lo + (s - c.rem), it);
            }
            if (c.ns > 1) row += c.ns * R * hkv;
        }
    }
    __syncthreads();

    // 3b. tensor-core items, longest key range first (counting sort on the
    // number of 128-key tiles), so persistent CTAs that take items in order
    // finish together.
    if (total_qtiles > 0) {
        for (int i = tid; i < kSortBins; i += kT) bins[i] = 0;
        // the longest tensor-core item: a request's last query tile
        int max_tiles = 0;
        for (int b = tid; b < p.num_seqs; b += kT) {
            const ReqInfo r = req(b);
            if (r.qtiles > 0) max_tiles = max(max_tiles, long_tiles(p, r, r.qtiles - 1));
        }
        {
            long long unused[1] = {0};
            block_reduce<kT, 1>(unused, max_tiles, tmpl);
        }
        const int shift_l = bin_shift(max_tiles, kSortBins);
        for (int b = tid; b < p.num_seqs; b += kT) {
            const ReqInfo r = req(b);
            for (int qt = 0; qt < r.qtiles; ++qt)
                atomicAdd(&bins[len_bin(long_tiles(p, r, qt), shift_l, kSortBins)], 1);
        }
        __syncthreads();
        {
            // one bin per thread: exclusive scan gives each bin's first slot
            int tot_l;
            const int v = tid < kSortBins ? bins[tid] : 0;
            const int off = block_exclusive_scan<kT>(v, tmp, &tot_l);
            if (tid < kSortBins) bins[tid] = off;
            long_base = tot_l;
            __syncthreads();
        }
        if (static_cast<long long>(long_base) * hkv > p.max_long) {
            if (tid == 0) s_overflow = 1;
        } else {
            for (int b = tid; b < p.num_seqs; b += kT) {
                const ReqInfo r = req(b);
                for (int qt = 0; qt < r.qtiles; ++qt) {
                    const int nvalid = min(p.q_tile_tokens, r.n - qt * p.q_tile_tokens);
                    LongItem it{};
                    it.b = b;
                    it.q_tile = qt;
                    it.key_begin = 0;
                    it.key_end = min(r.len, r.ctx + qt * p.q_tile_tokens + nvalid);
                    store_record(p.long_items,
                                 atomicAdd(&bins[len_bin(long_tiles(p, r, qt), shift_l,
                                                         kSortBins)], 1),
                                 it);
                }
            }
        }
    }

    // 4. counters and header ----------------------------------------------------
    for (int i = tid; i < p.num_counters; i += kT) p.counters[i] = 0;
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
    if (p.num_seqs <= kSmallPlanSeqs) {
        PdlLaunch l(1, 32, 0, s);
        return launch_kernel(l, plan_kernel<32>, p) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    PdlLaunch l(1, kPlanThreads, 0, s);
    return launch_kernel(l, plan_kernel<kPlanThreads>, p) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
