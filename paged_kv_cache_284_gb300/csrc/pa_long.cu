// pa_long.cu -- tensor-core attention for long query rows: chunked-prefill
// chunks, prefix-cache hits and whole prompts ("vLLM中如何实现大模型推理加速
// 技术？": chunked prefill / prefix caching; "11. 推理加速(一):vLLM 原理",
// §11.3: prefill is compute-bound), and the cascade shared-prefix pass
// (2048ai.net page on the vLLM V1 engine, §02.1 级联推理: one multi-query
// pass over the shared KV, each prefix tile read once per 128 query rows).
//
// One persistent CTA per SM walks its share of the work items (128-row query
// tile x key range), FlashAttention style, on the 5th-generation tensor cores:
//  * rows of a tile are (token, head) pairs of one kv head's GQA group:
//    128 / group tokens x group heads, loaded by one 3-D TMA box per 64 dims;
//  * warp 0 gathers 128-key K tiles through the block table (eight 16-key TMA
//    boxes, 128-byte swizzle) into a 2-deep ring that is released as soon as
//    S = Q K^T has consumed it; warp 10 does the same for V into a 3-deep ring
//    released after O += P V;
//  * warp 1 issues tcgen05.mma S = Q K^T (M=128, N=128, K=head_dim) into one
//    of two TMEM S buffers as soon as K and a buffer are free; warp 11 issues
//    O += P V (M=128, N=head_dim, K=128) as soon as P is ready, into a
//    TMEM O accumulator, with P read from TMEM and V read N-major straight
//    from its cache layout;
//  * warps 2-9 (two threads per row, one per half of its 128 keys) read S from TMEM, apply the
//    context-offset causal mask (row i of a request with context c sees keys
//    0..c+i), run the online softmax in the log2 domain with a lazy max
//    update, rescale O in TMEM only when the max grows by more than 2^8, and
//    write P (bf16) into one of two TMEM P buffers; P V trails Q K^T by two
//    tiles so the tensor cores always have the next scores to compute;
//  * the epilogue reads O from TMEM, normalises and stores bf16 (or, for a
//    split prefix, fp32 split states that prefix_fold_kernel merges with the
//    merge operator) while the next item's Q, K and V are already streaming
//    in.
// Key tiles entirely above a tile's causal limit are never visited.
#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kKStages = 2;  // K is released as soon as Q K^T has read it
constexpr int kVStages = 3;  // V is held until the P V two tiles later
// warps: 0 K (+Q) loads, 1 Q K^T issuer (+TMEM allocation), 2-9 softmax, 10 V loads,
// 11 P V issuer
constexpr int kLongWarps = 12;
constexpr int kWarpV = 10, kWarpPV = 11;
constexpr int kSoftmaxWarps = 8;

template <int D>
struct LongGeom {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = 128 * 128;            // 128 rows x 128 B
    static constexpr int kQBytes = kHalves * kHalfBytes;    // Q tile
    static constexpr int kKVBytes = kHalves * kHalfBytes;   // one K (or V) tile of 128 keys
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKVBytes;
    static constexpr int kOffBar = kOffV + kVStages * kKVBytes;
    static constexpr int kCtlBytes = 512;
    // row-half exchange: partial maxima [2 tile parities][2 halves][128 rows]
    // and partial sums [2 halves][128 rows]
    static constexpr int kOffXchg = kOffBar + kCtlBytes;
    static constexpr int kXchgBytes = (2 * 2 * 128 + 2 * 128) * 4;
    // dynamic schedule: published item indices, their count, and how many
    // each warp has read
    static constexpr int kOffQueue = kOffXchg + kXchgBytes;
    static constexpr int kQueueBytes = 512;
    // at least 116 KiB so that one CTA owns an SM (and its 512 TMEM columns)
    static constexpr int kSmemRaw = kOffQueue + kQueueBytes + 1024;
    static constexpr int kSmemBytes = kSmemRaw > 116 * 1024 ? kSmemRaw : 116 * 1024;
    // TMEM columns: S0 | S1 (fp32 scores) | O (fp32) | P0 | P1 (bf16 pairs)
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kColS = 0, kColO = 2 * kLongKeys, kColP = 3 * kLongKeys;
    static_assert(kColO + D <= kColP, "O overlaps P");
};

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[2];  // by tile parity: a softmax half may run a tile ahead
    uint64_t pv_done[2];  // P V of a tile finished, by the tile's P buffer
    uint64_t xchg[4];  // row-half exchange, one per TMEM lane quarter (2 warps each)
    uint64_t o_free, drain, drain_pv;
};

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return warp_mbar_wait(bar, parity, abort);
}

// Packed pairs of fp32 (one 64-bit register pair) for the two-wide FMA / add
// of this architecture, and the three-input maximum: the softmax warps are
// bound by instruction issue, so each score costs half an FMA, half an add,
// half a conversion, half a maximum and one exponential.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Everything one role needs to know about a work item.
struct Item {
    int b, h, tok0, nvalid, pos0, key_begin, key_end, causal, nsplit, split;
    int pair, partial_base, nt;
};

__device__ __forceinline__ Item decode_item(const LongParams &p, int idx) {
    Item it{};
    const int TQ = p.q_tile_tokens;
    if (!p.prefix_mode) {
        const int rec = idx / p.num_kv_heads;
        const LongItem li = load_record(p.items, rec);
        it.b = li.b;
        it.h = idx - rec * p.num_kv_heads;
        const int q0 = __ldg(p.qsl + li.b);
        const int n = __ldg(p.qsl + li.b + 1) - q0;
        it.tok0 = q0 + li.q_tile * TQ;
        it.nvalid = min(TQ, n - li.q_tile * TQ);
        it.pos0 = __ldg(p.ctx + li.b) + li.q_tile * TQ;
        it.key_begin = li.key_begin;
        it.key_end = li.key_end;
        it.causal = 1;
        it.nsplit = 1;
    } else {
        it.split = idx % p.prefix_nsplit;
        const int qt = (idx / p.prefix_nsplit) % p.prefix_q_tiles;
        it.h = idx / (p.prefix_nsplit * p.prefix_q_tiles);
        it.nsplit = p.prefix_nsplit;
        it.tok0 = qt * TQ;
        it.nvalid = min(TQ, p.num_q_tokens - it.tok0);
        it.key_begin = it.split * p.prefix_split_keys;
        it.key_end = min(p.prefix_len, it.key_begin + p.prefix_split_keys);
        it.pair = it.h * p.prefix_q_tiles + qt;
        it.partial_base = it.pair * it.nsplit * kLongRows;
    }
    const int span = it.key_end - it.key_begin;
    it.nt = span > 0 ? (span + kLongKeys - 1) / kLongKeys : 0;
    return it;
}

// Item a CTA takes in round k: items are sorted longest first, and the CTAs
// take them in serpentine order (left to right, then right to left), which
// keeps the per-CTA totals close to a longest-processing-time schedule.
__device__ __forceinline__ int serpentine_item(int round) {
    const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return round * g + ((round & 1) ? g - 1 - c : c);
}

// Dynamic schedule (p.dynamic): warp 0 -- the K producer, which runs ahead
// of every other role -- takes item indices from the step's counter, shared
// by every launch of the step, and publishes them in order in a shared
// memory queue; every other warp reads them back in the same order.  A
// CTA that starts late therefore simply takes fewer items.
constexpr int kItemQueue = 64;
constexpr int kSchedDone = -1, kSchedAbort = -2;
struct Sched {
    int *idx;            // [kItemQueue]
    volatile int *pub;   // items published
    volatile int *cons;  // [kLongWarps] items read per warp
};

__device__ __forceinline__ bool sched_spin(bool (*ready)(const Sched &, int), const Sched &sc,
                                           int k, volatile int *abort) {
    if (ready(sc, k)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (ready(sc, k)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            *abort = 1;
            return false;
        }
    }
}
__device__ bool sched_published(const Sched &sc, int k) { return *sc.pub > k; }
__device__ bool sched_slot_free(const Sched &sc, int k) {
    for (int w = 1; w < kLongWarps; ++w)
        if (sc.cons[w] <= k - kItemQueue) return false;
    return true;
}

// Item of round k of this role, or kSchedDone / kSchedAbort.  One thread of
// the warp calls it (a whole-warp role broadcasts the result).
__device__ __forceinline__ int sched_take(const LongParams &p, const Sched &sc, int n_items,
                                          int k, int warp, volatile int *abort) {
    if (!p.dynamic) {
        if (k * static_cast<int>(gridDim.x) >= n_items) return kSchedDone;
        const int idx = serpentine_item(k);
        return idx < n_items ? idx : kSchedDone;
    }
    const int slot = k % kItemQueue;
    int idx;
    if (warp == 0) {
        if (k >= kItemQueue && !sched_spin(sched_slot_free, sc, k, abort)) return kSchedAbort;
        idx = atomicAdd(&p.hdr->long_next, 1);
        if (idx >= n_items) idx = kSchedDone;
        sc.idx[slot] = idx;
        __threadfence_block();
        *sc.pub = k + 1;
    } else {
        if (!sched_spin(sched_published, sc, k, abort)) return kSchedAbort;
        __threadfence_block();
        idx = reinterpret_cast<volatile int *>(sc.idx)[slot];
        sc.cons[warp] = k + 1;
    }
    return idx;
}

__device__ __forceinline__ int num_items(const LongParams &p) {
    if (p.prefix_mode) return p.num_kv_heads * p.prefix_q_tiles * p.prefix_nsplit;
    return *reinterpret_cast<volatile int *>(&p.hdr->num_long_items);
}

// Producer loop shared by the K warp (0, which also loads Q) and the V warp
// (6): gathers one 128-key tile per step into its ring.
template <int D, int NS>
__device__ void produce(const LongParams &p, const Sched &sc, const CUtensorMap *tm, uint8_t *ring,
                        uint64_t *full, uint64_t *empty, Bars *bars, bool load_q,
                        const CUtensorMap *tmq, uint8_t *sQ, volatile int *abort_flag) {
    using G = LongGeom<D>;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_items = num_items(p);
    uint32_t t = 0;        // tiles issued by this warp so far (all items)
    uint32_t k_item = 0;   // items (with keys) started so far
    bool ok = true;
    for (int round = 0; ok; ++round) {
        int idx = 0;
        if (lane == 0) idx = sched_take(p, sc, n_items, round, warp, abort_flag);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx == kSchedDone) break;
        if (idx == kSchedAbort) {
            ok = false;
            break;
        }
        const Item it = decode_item(p, idx);
        if (it.nt == 0) continue;
        if (load_q) {
            if (k_item > 0 && !warp_wait(&bars->q_empty, (k_item - 1) & 1, abort_flag)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->q_full,
                                      static_cast<uint32_t>(G::kHalves * 128 * p.group *
                                                            p.q_tile_tokens));
                for (int hf = 0; hf < G::kHalves; ++hf)
                    tma_load_3d(sQ + hf * G::kHalfBytes, tmq, hf * 64, it.h * p.group, it.tok0,
                                &bars->q_full);
            }
        }
        ++k_item;
        const int *bt = p.block_tables + static_cast<int64_t>(it.b) * p.bt_stride;
        int my_row = p.kv_rows;
        for (int j = 0; j < it.nt; ++j, ++t) {
            if ((j & 3) == 0) {
                // rows of the next 32 chunks (4 tiles), one per lane; chunks
                // past key_end are read fully out of bounds -> zeros
                const int key0 = it.key_begin + (j * 8 + lane) * kChunkKeys;
                my_row = p.kv_rows;
                if (key0 < it.key_end) {
                    int col = key0 / p.block_size;
                    if (p.bt_stride > 0 && col >= p.bt_stride) {
                        flag_status(p.status, PA_DEV_BAD_METADATA);
                        col = p.bt_stride - 1;
                    }
                    // fp8 pool: block col of a staged request is its staging block
                    int blk = p.stage_base ? __ldcg(p.stage_base + it.b) + col : __ldg(bt + col);
                    if (blk < 0 || blk >= p.num_blocks) {
                        flag_status(p.status, PA_DEV_BAD_BLOCK);
                        blk = min(max(blk, 0), p.num_blocks - 1);
                    }
                    my_row = (blk * p.num_kv_heads + it.h) * p.block_size + key0 % p.block_size;
                }
            }
            const int slot = t % NS;
            if (t >= NS && !warp_wait(&empty[slot], ((t / NS) - 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(G::kKVBytes));
            __syncwarp();
            const int c = lane & 7;
            const int row = __shfl_sync(0xffffffffu, my_row, (j & 3) * 8 + c);
            if (lane < 8) {
#pragma unroll
                for (int hf = 0; hf < G::kHalves; ++hf)
                    tma_load_2d(ring + slot * G::kKVBytes + hf * G::kHalfBytes + c * 2048, tm,
                                hf * 64, row, &full[slot]);
            }
            __syncwarp();
        }
    }
    if (*abort_flag && lane == 0) {
        // let copies already in flight land before the CTA exits
        for (uint32_t k = (t > NS ? t - NS : 0); k < t; ++k) mbar_drain(&full[k % NS], (k / NS) & 1);
    }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(32 * kLongWarps, 1)
    long_kernel(const LongParams p, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using G = LongGeom<D>;
    constexpr int KS = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + G::kOffBar);
    int *ctl = reinterpret_cast<int *>(smem + G::kOffBar + 256);
    volatile int *abort_flag = ctl;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (p.wait_start) {
        pdl_wait();     // the plan (and any staging copy) first
        pdl_trigger();  // then the split-KV grid may take the other SMs
    }
    const int n_items = num_items(p);
    if (!p.dynamic && static_cast<int>(blockIdx.x) >= n_items) {
        pdl_wait();  // complete only after the grid this one overlaps
        return;
    }
    int *qmem = reinterpret_cast<int *>(smem + G::kOffQueue);
    Sched sched;
    sched.idx = qmem;
    sched.pub = qmem + kItemQueue;
    sched.cons = qmem + kItemQueue + 1;

    // ---- setup ----------------------------------------------------------------
    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        mbar_init(&bars->q_empty, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&bars->k_full[i], 1);
            mbar_init(&bars->k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], kSoftmaxWarps);
        }
        mbar_init(&bars->p_full[0], kSoftmaxWarps);
        mbar_init(&bars->p_full[1], kSoftmaxWarps);
        mbar_init(&bars->pv_done[0], 1);
        mbar_init(&bars->pv_done[1], 1);
        mbar_init(&bars->o_free, kSoftmaxWarps);
        for (int i = 0; i < 4; ++i) mbar_init(&bars->xchg[i], 2);
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->drain_pv, 1);
        ctl[0] = 0;
        *sched.pub = 0;
        for (int w = 0; w < kLongWarps; ++w) sched.cons[w] = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, G::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    uint8_t *sQ = smem + G::kOffQ;
    uint8_t *sK = smem + G::kOffK;
    uint8_t *sV = smem + G::kOffV;

    if (warp == 0) {
        // ============================ K (and Q) loads ============================
        if (lane == 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
        }
        produce<D, kKStages>(p, sched, &tmk, sK, bars->k_full, bars->k_empty, bars, true, &tmq, sQ,
                             abort_flag);
    } else if (warp == kWarpV) {
        // ============================ V loads ============================
        if (lane == 0) tma_prefetch_desc(&tmv);
        produce<D, kVStages>(p, sched, &tmv, sV, bars->v_full, bars->v_empty, bars, false, nullptr,
                             nullptr, abort_flag);
    } else if (warp == 1) {
        // ============================ Q K^T issuer ============================
        // Runs ahead of the softmax: a tile's scores only wait for its K tile and
        // for the softmax to have read the scores two tiles back.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kLongRows, kLongKeys, 0);
            const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK);
            uint32_t t = 0, k_item = 0;
            bool ok = true;
            for (int round = 0; ok; ++round) {
                const int idx = sched_take(p, sched, n_items, round, warp, abort_flag);
                if (idx == kSchedDone) break;
                if (idx == kSchedAbort) {
                    ok = false;
                    break;
                }
                const Item it = decode_item(p, idx);
                if (it.nt == 0) continue;
                if (!mbar_wait(&bars->q_full, k_item & 1, abort_flag)) { ok = false; break; }
                int j = 0;
                for (; j < it.nt; ++j) {
                    const uint32_t tt = t + j;
                    const int ks = tt % kKStages;
                    const int sb = tt & 1;
                    if (!mbar_wait(&bars->k_full[ks], (tt / kKStages) & 1, abort_flag)) { ok = false; break; }
                    if (tt >= 2 && !mbar_wait(&bars->s_free[sb], ((tt - 2) >> 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kb = k_addr + ks * G::kKVBytes;
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint64_t ad = smem_desc_sw128(
                            q_addr + (kk >> 2) * G::kHalfBytes + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(
                            kb + (kk >> 2) * G::kHalfBytes + (kk & 3) * 32, 16, 1024);
                        tc_mma(tmem + G::kColS + sb * kLongKeys, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&bars->k_empty[ks]);
                    tc_commit(&bars->s_full[sb]);
                    if (j == it.nt - 1) tc_commit(&bars->q_empty);
                }
                if (p.tile_counter) atomicAdd(p.tile_counter, static_cast<unsigned long long>(j));
                t += it.nt;
                ++k_item;
            }
            if (!ok) {
                // let every MMA already issued finish before TMEM is released
                tc_commit(&bars->drain);
                mbar_drain(&bars->drain, 0);
            }
        }
    } else if (warp == kWarpPV) {
        // ============================ P V issuer ============================
        // Follows the softmax: a tile's P V waits for its P, its V tile and, at
        // the start of an item, for the previous item's epilogue to read O.
        if (lane == 0) {
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kLongRows, D, 1);
            const uint32_t v_addr = smem_u32(sV);
            uint32_t t = 0, k_item = 0;
            bool ok = true;
            for (int round = 0; ok; ++round) {
                const int idx = sched_take(p, sched, n_items, round, warp, abort_flag);
                if (idx == kSchedDone) break;
                if (idx == kSchedAbort) {
                    ok = false;
                    break;
                }
                const Item it = decode_item(p, idx);
                if (it.nt == 0) continue;
                for (int j = 0; j < it.nt; ++j) {
                    const uint32_t tt = t + j;
                    if (!mbar_wait(&bars->p_full[tt & 1], (tt >> 1) & 1, abort_flag)) { ok = false; break; }
                    if (j == 0 && k_item > 0 &&
                        !mbar_wait(&bars->o_free, (k_item - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int vs = tt % kVStages;
                    if (!mbar_wait(&bars->v_full[vs], (tt / kVStages) & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t vbase = v_addr + vs * G::kKVBytes;
                    // P (bf16) of this tile: row r in TMEM lane r, key k in column k / 2
                    const uint32_t pcol = tmem + G::kColP + (tt & 1) * (kLongKeys / 2);
#pragma unroll
                    for (int kk = 0; kk < kLongKeys / 16; ++kk) {
                        const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, G::kHalfBytes, 1024);
                        tc_mma_ts(tmem + G::kColO, pcol + kk * 8, bd, idesc_pv,
                                  (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&bars->v_empty[vs]);
                    tc_commit(&bars->pv_done[tt & 1]);
                }
                t += it.nt;
                ++k_item;
            }
            if (!ok) {
                tc_commit(&bars->drain_pv);
                mbar_drain(&bars->drain_pv, 0);
            }
        }
    } else {
        // ============================ softmax + epilogue ============================
        // Two warps per TMEM lane quarter: warps 2-5 own columns 0-63 of their
        // rows, warps 6-9 columns 64-127.  The two halves of a row swap their
        // partial maxima through spare TMEM columns each tile and add their
        // partial sums once per item.
        const int wq = warp & 3;  // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;
        const int r = wq * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const int ttok = r / p.group;
        const int jh = r - ttok * p.group;
        const int c0 = half * (kLongKeys / 2);  // first S / P column of this half
        const int o0 = half * (D / 2);          // first O column of this half
        uint32_t t = 0, x_phase = 0;
        bool ok = true;
        // swap one float with the other half of the row (same row, other warp)
        float *xch = reinterpret_cast<float *>(smem + G::kOffXchg);
        auto swap_halves = [&](float *slots, float mine, float &theirs) -> bool {
            slots[half * 128 + r] = mine;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->xchg[wq]);
            const bool w = warp_wait(&bars->xchg[wq], x_phase & 1, abort_flag);
            ++x_phase;
            theirs = slots[(1 - half) * 128 + r];
            return w;
        };
        for (int round = 0; ok; ++round) {
            int idx = 0;
            if (lane == 0) idx = sched_take(p, sched, n_items, round, warp, abort_flag);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (idx == kSchedDone) break;
            if (idx == kSchedAbort) {
                ok = false;
                break;
            }
            const Item it = decode_item(p, idx);
            const bool row_valid = ttok < it.nvalid && r < p.q_tile_tokens * p.group;
            const int row_limit = it.causal ? it.pos0 + ttok : 0x7fffffff;
            const int tile_limit_min = it.causal ? it.pos0 : 0x7fffffff;
            float m_used = -INFINITY, l = 0.f;
            // scores in log2 units; an fp8 pool's K scale folds in here
            const float sl2 = p.k_scale ? p.scale_log2 * __ldg(p.k_scale + it.h) : p.scale_log2;
            for (int j = 0; ok && j < it.nt; ++j) {
                const uint32_t tt = t + j;
                const int sb = tt & 1;
                if (!warp_wait(&bars->s_full[sb], (tt >> 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                uint32_t s0[32], s1[32];
                const uint32_t sa = t_lane + G::kColS + sb * kLongKeys + c0;
                tmem_ld32(sa, s0);
                tmem_ld32(sa + 32, s1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_free[sb]);
                const int kb = it.key_begin + j * kLongKeys;
                const bool need_mask =
                    (kb + kLongKeys - 1 > tile_limit_min) || (kb + kLongKeys > it.key_end);
                if (need_mask) {
                    // keys [0, lim) of this half are visible to this row
                    const int lim = min(row_limit, it.key_end - 1) - (kb + c0) + 1;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (i >= lim) s0[i] = __float_as_uint(-INFINITY);
                        if (32 + i >= lim) s1[i] = __float_as_uint(-INFINITY);
                    }
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    mx0 = max3(mx0, __uint_as_float(s0[i]), __uint_as_float(s0[i + 1]));
                    mx1 = max3(mx1, __uint_as_float(s0[16 + i]), __uint_as_float(s0[17 + i]));
                    mx2 = max3(mx2, __uint_as_float(s1[i]), __uint_as_float(s1[i + 1]));
                    mx3 = max3(mx3, __uint_as_float(s1[16 + i]), __uint_as_float(s1[17 + i]));
                }
                float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                float other;
                if (!swap_halves(xch + (tt & 1) * 256, mx, other)) { ok = false; break; }
                mx = fmaxf(mx, other);
                const float mxs = mx * sl2;  // scale > 0: max commutes with it
                float alpha = 1.f;
                if (mxs > m_used + kRescaleThreshold || (m_used == -INFINITY && mxs > -INFINITY)) {
                    alpha = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mxs);
                    m_used = mxs;
                }
                const float neg_ref = m_used == -INFINITY ? 0.f : -m_used;
                // this half's 64 keys of P row r (bf16 pairs) go to the tile's TMEM
                // P buffer, the A operand of its P V, in two 32-key pieces so the
                // first store overlaps the second piece's exponentials; the P V
                // that used this buffer two tiles ago must be done
                if (tt >= 2 && !warp_wait(&bars->pv_done[sb], ((tt - 2) >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pdst = t_lane + G::kColP + sb * (kLongKeys / 2) + half * 32;
                const uint64_t sc2 = f2_pack(sl2, sl2);
                const uint64_t nr2 = f2_pack(neg_ref, neg_ref);
                uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
                for (int piece = 0; piece < 2; ++piece) {
                    const uint32_t *sv = piece ? s1 : s0;
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        float a0, a1, a2, a3;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                                         sc2, nr2), a0, a1);
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * i + 2]), __uint_as_float(sv[2 * i + 3])),
                                         sc2, nr2), a2, a3);
                        a0 = fast_exp2(a0);
                        a1 = fast_exp2(a1);
                        a2 = fast_exp2(a2);
                        a3 = fast_exp2(a3);
                        acc0 = f2_add(acc0, f2_pack(a0, a1));
                        acc1 = f2_add(acc1, f2_pack(a2, a3));
                        pk[i] = pack_bf16x2(a0, a1);
                        pk[i + 1] = pack_bf16x2(a2, a3);
                    }
                    tmem_st16(pdst + piece * 16, pk);
                }
                float sum0, sum1, sum2, sum3;
                f2_unpack(acc0, sum0, sum1);
                f2_unpack(acc1, sum2, sum3);
                l = l * alpha + ((sum0 + sum1) + (sum2 + sum3));
                if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // O is rescaled in place: the previous tile's P V must be done
                    if (!warp_wait(&bars->pv_done[(tt - 1) & 1], ((tt - 1) >> 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t raw[32];
#pragma unroll
                    for (int qd = 0; qd < D / 64; ++qd) {
                        tmem_ld32(t_lane + G::kColO + o0 + qd * 32, raw);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
                        tmem_st32(t_lane + G::kColO + o0 + qd * 32, raw);
                    }
                    tmem_wait_st();
                }
                if (kb + kLongKeys > it.key_end) {
                    // the last loaded chunk may extend past the keys: zero those V
                    // rows so 0-probabilities never meet non-finite cache contents
                    const int vs = tt % kVStages;
                    if (!warp_wait(&bars->v_full[vs], (tt / kVStages) & 1, abort_flag)) { ok = false; break; }
                    const int z0 = it.key_end - kb;                  // first row to clear
                    const int z1 = min(kLongKeys, (z0 + 15) & ~15);  // end of its chunk
                    const int pieces = (z1 - z0) * 8 * G::kHalves;   // 16-byte pieces
                    for (int q = r + half * 128; q < pieces; q += 256) {
                        const int hf = q / ((z1 - z0) * 8);
                        const int rem = q - hf * (z1 - z0) * 8;
                        const int row = z0 + rem / 8, piece = rem % 8;
                        *reinterpret_cast<uint4 *>(sV + vs * G::kKVBytes + hf * G::kHalfBytes +
                                                   row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                tmem_wait_st();
                if (kb + kLongKeys > it.key_end) fence_proxy_async_smem();  // zeroed V rows
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_full[sb]);
            }
            if (ok && it.nt > 0) {
                const uint32_t last = t + it.nt - 1;
                ok = warp_wait(&bars->pv_done[last & 1], (last >> 1) & 1, abort_flag);
            }
            tc_fence_after();
            if (ok && it.nt > 0) {
                float l_other = 0.f;
                ok = swap_halves(xch + 512, l, l_other);
                l += l_other;
            }

            // ---- epilogue of this item: this half's D/2 output columns ----
            // an fp8 pool's V scale multiplies the output
            const float vsc = p.v_scale ? __ldg(p.v_scale + it.h) : 1.f;
            const float inv = l > 0.f ? vsc / l : 0.f;
            const float lse_v = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
            const int tok = it.tok0 + ttok;
            const int hq = it.h * p.group + jh;
            const int64_t orow = static_cast<int64_t>(tok) * p.num_q_heads + hq;
            const bool direct = it.nsplit == 1 && !p.states_only;
            const int64_t prow = static_cast<int64_t>(it.partial_base + it.split * kLongRows + r);
            for (int qd = 0; qd < D / 64; ++qd) {
                const int col = o0 + qd * 32;
                uint32_t raw[32];
                if (ok && it.nt > 0) {
                    tmem_ld32(t_lane + G::kColO + col, raw);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) raw[i] = 0u;
                }
                if (!ok || !row_valid) continue;
                if (direct && !p.out_f32) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + col);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 0]) * inv, __uint_as_float(raw[v4 * 8 + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 2]) * inv, __uint_as_float(raw[v4 * 8 + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 4]) * inv, __uint_as_float(raw[v4 * 8 + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 6]) * inv, __uint_as_float(raw[v4 * 8 + 7]) * inv);
                        dst[v4] = w;
                    }
                } else {
                    float *dst = direct ? p.out_f32 + orow * D + col : p.partial_o + prow * D + col;
#pragma unroll
                    for (int v4 = 0; v4 < 8; ++v4)
                        __stcg(reinterpret_cast<float4 *>(dst) + v4,
                               make_float4(__uint_as_float(raw[v4 * 4 + 0]) * inv, __uint_as_float(raw[v4 * 4 + 1]) * inv,
                                           __uint_as_float(raw[v4 * 4 + 2]) * inv, __uint_as_float(raw[v4 * 4 + 3]) * inv));
                }
            }
            // O has been read: the next item's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (it.nt > 0 && lane == 0) mbar_arrive(&bars->o_free);
            if (ok && row_valid && half == 0) {
                if (direct) {
                    if (p.lse) p.lse[orow] = lse_v;
                } else {
                    __stcg(p.partial_lse + prow, lse_v);
                }
            }
            t += it.nt;
        }
    }

    if (*abort_flag && threadIdx.x == 0) flag_status(p.status, PA_DEV_WAIT_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, G::kTmemCols);
    // with overlap_prev: this grid completes only after the split-KV grid it
    // overlapped, so later work on the stream is still ordered after both
    pdl_wait();
    if (p.first_done && threadIdx.x == 0) {
        if (p.first_ctas < 0) {
            // a first launch of the step: count this CTA done (its outputs first)
            __threadfence();
            atomicAdd(p.first_done, 1);
        } else {
            // the last launch: complete only after every CTA of the first one
            const uint64_t t0 = global_timer_ns();
            while (*reinterpret_cast<volatile int *>(p.first_done) < p.first_ctas) {
                if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                    flag_status(p.status, PA_DEV_WAIT_TIMEOUT);
                    break;
                }
            }
            __threadfence();
        }
    }
}

// Merge of the prefix pass's split states with the merge operator (2048ai.net
// page on the vLLM V1 engine, §02.1 级联推理): one warp per query row of a
// (kv head, query tile), its lanes across the head dimension, so that all
// splits' loads of a row are in flight at once and the work spreads over
// many SMs (one CTA per 8 rows).  A split count of at most 64 is assumed.
// With f.extra_o set, one more state per row (cascade decode's unique-suffix
// state) joins the merge: the prefix and suffix halves of cascade inference
// meet here, in one epilogue.
template <int D>
__global__ void __launch_bounds__(256) prefix_fold_kernel(const PrefixFoldParams f) {
    pdl_wait();  // the prefix pass's states
    const int lane = threadIdx.x & 31;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int pair = static_cast<int>(w / kLongRows), r = static_cast<int>(w % kLongRows);
    if (pair >= f.pairs || r >= f.q_tile_tokens * f.group) return;
    const int ttok = r / f.group, jh = r - ttok * f.group;
    const int h = pair / f.q_tiles, qt = pair - h * f.q_tiles;
    const int tok = qt * f.q_tile_tokens + ttok;
    if (tok >= f.num_q_tokens) return;
    const int ns = f.nsplit;
    const int64_t base = static_cast<int64_t>(pair) * ns * kLongRows + r;
    // split s's log-sum-exp lives in lane s % 32, slot s / 32
    const float l0 = lane < ns ? __ldcg(f.partial_lse + base + lane * kLongRows) : -INFINITY;
    const float l1 = lane + 32 < ns ? __ldcg(f.partial_lse + base + (lane + 32) * kLongRows)
                                    : -INFINITY;
    const int64_t row = static_cast<int64_t>(tok) * f.num_q_heads + h * f.group + jh;
    const float xl = f.extra_o ? __ldcg(f.extra_lse + row) : -INFINITY;
    float M = fmaxf(fmaxf(l0, l1), xl);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w0 = (lane < ns && M != -INFINITY) ? __expf(l0 - M) : 0.f;
    const float w1 = (lane + 32 < ns && M != -INFINITY) ? __expf(l1 - M) : 0.f;
    const float wx = (xl != -INFINITY) ? __expf(xl - M) : 0.f;
    float wsum = w0 + w1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    wsum += wx;
    const bool col = lane < D / 4;  // this lane's float4 of the row
    const float4 *po = reinterpret_cast<const float4 *>(f.partial_o + base * D) + (col ? lane : 0);
    const int64_t stride = static_cast<int64_t>(kLongRows) * (D / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (wx > 0.f && col) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(f.extra_o + row * D) + lane);
        acc = make_float4(wx * v.x, wx * v.y, wx * v.z, wx * v.w);
    }
    for (int s0 = 0; s0 < ns; s0 += 8) {
        float ws[8];
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int s = s0 + j;
            const float a = __shfl_sync(0xffffffffu, w0, s & 31);
            const float b = __shfl_sync(0xffffffffu, w1, s & 31);
            ws[j] = s < ns ? (s < 32 ? a : b) : 0.f;
            v[j] = (col && s < ns) ? __ldcg(po + s * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc.x += ws[j] * v[j].x;
            acc.y += ws[j] * v[j].y;
            acc.z += ws[j] * v[j].z;
            acc.w += ws[j] * v[j].w;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (col) {
        const float4 a = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (f.out_f32) {
            reinterpret_cast<float4 *>(f.out_f32 + row * D)[lane] = a;
        } else {
            uint2 pk2;
            pk2.x = pack_bf16x2(a.x, a.y);
            pk2.y = pack_bf16x2(a.z, a.w);
            reinterpret_cast<uint2 *>(f.out + row * D)[lane] = pk2;
        }
    }
    if (lane == 0 && f.lse) f.lse[row] = wsum > 0.f ? M + __logf(wsum) : -INFINITY;
}

int launch_prefix_fold(const PrefixFoldParams &f, int head_dim, cudaStream_t s) {
    const int64_t warps = static_cast<int64_t>(f.pairs) * kLongRows;
    const unsigned grid = static_cast<unsigned>((warps + 7) / 8);
    if (grid == 0) return PA_OK;
    PdlLaunch l(grid, 256, 0, s);
    const cudaError_t e = head_dim == 128 ? launch_kernel(l, prefix_fold_kernel<128>, f)
                                          : launch_kernel(l, prefix_fold_kernel<64>, f);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t long_smem_bytes(int head_dim) {
    return head_dim == 128 ? LongGeom<128>::kSmemBytes : LongGeom<64>::kSmemBytes;
}

template <int D>
static int configure_long() {
    static PerDeviceOnce once;
    return once_per_device(once, [] {
        return cudaFuncSetAttribute(long_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    LongGeom<D>::kSmemBytes);
    });
}

// grid: the caller passes an upper bound on the number of items; the kernel is
// persistent, so at most one CTA per SM is launched.
int launch_long(const LongParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                const CUtensorMap &tv, int head_dim, int grid, cudaStream_t s) {
    if (grid <= 0) return PA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    grid = grid < sms ? grid : sms;
    const bool pdl = p.overlap_prev != 0 || p.wait_start != 0;
    if (head_dim == 128) {
        if (configure_long<128>() != PA_OK) return PA_ERR_CUDA;
        PdlLaunch l(grid, 32 * kLongWarps, LongGeom<128>::kSmemBytes, s, pdl);
        return launch_kernel(l, long_kernel<128>, p, tq, tk, tv) == cudaSuccess
                   ? PA_OK
                   : PA_ERR_CUDA;
    }
    if (configure_long<64>() != PA_OK) return PA_ERR_CUDA;
    PdlLaunch l(grid, 32 * kLongWarps, LongGeom<64>::kSmemBytes, s, pdl);
    return launch_kernel(l, long_kernel<64>, p, tq, tk, tv) == cudaSuccess ? PA_OK
                                                                                    : PA_ERR_CUDA;
}

}  // namespace pa
