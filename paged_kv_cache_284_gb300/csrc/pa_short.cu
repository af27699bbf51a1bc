// pa_short.cu -- split-KV attention for short query rows: decode (q_len 1),
// speculative verify (q_len 1 + k) and small chunks, i.e. every request whose
// q_len * group fits 64 rows.  This is the memory-bound half of the step
// ("11. 推理加速(一):vLLM 原理", §11.3: decode is memory-bound; "PagedAttention
// (with_kvcache)").
//
// Design (one persistent CTA per SM slot, 5 warps):
//  * warp 4 is the producer: it pulls work items (request b, kv head h, key
//    range) from a device counter, turns the block table into TMA row
//    coordinates 32 chunks at a time (one lane per chunk), and four lanes
//    issue the TMA tensor loads (128-byte swizzled boxes of 16 keys x 64
//    dims) of a stage's four chunks of K and V at once, into a 3-deep ring
//    of 64-key stages.  The ring keeps running across item boundaries.
//  * warps 0-3 consume: for each 16-key chunk, S = Q K^T and O += P V on
//    mma.sync (bf16 in, fp32 accumulate) with an online softmax in the
//    log2 domain.  All g query heads of a kv head (and all q_len rows) are
//    rows of one 16..64-row tile, so every K/V byte is loaded once for the
//    whole GQA group.  With <= 16 rows the four warps split each stage's keys
//    and merge their states at the end of the item through the stage buffer.
//  * split-KV: a long sequence is cut into several items; each writes a
//    partial (o, lse) state, and the last item to finish (device counter)
//    folds them with the merge operator (2048ai.net page on the vLLM V1
//    engine, §02.1 级联推理) -- the fused split-KV epilogue.  For cascade
//    decode the final state of each row is written in fp32 instead, for the
//    fold that merges it with the shared-prefix state.
//  * FP8 pool (same page, §02 推理优化: KV-cache quantisation): K and V are
//    e4m3 codes, one 16-key x 128-dim TMA box per chunk (half the bytes of
//    bf16), 8 chunks (128 keys) per ring stage.  The MMAs run in f16: e4m3 decodes exactly to f16, q is
//    converted once per item, P is packed as f16.  K fragments come from
//    plain ldmatrix (each lane gets 4 consecutive dims of one key; q's dims
//    are permuted the same way inside each 16-dim k-step, which leaves the
//    dot products unchanged).  V fragments come from ldmatrix.trans over dim
//    pairs and a byte permute: each lane gets 2 keys x 2 dims, so the two
//    dims of a pair land in two different 8-column output tiles; the output
//    columns are permuted back when they are written.  Scores are scaled by
//    the kv head's K scale, outputs by its V scale.
//  * fp8 items with at most 8 rows (decode at group <= 8) swap the operands:
//    S^T = K Q^T puts the chunk's 16 keys on the MMA's M side and the rows on
//    N = 8, and O^T = V^T P^T puts 16 head dims on M, so a chunk takes 16
//    MMAs instead of 32 and each lane holds 2 keys x 2 rows.  P^T reaches
//    the second MMA's B operand through movmatrix (8x8 transposes).  The
//    row maximum is reduced across lanes only when some score exceeds the
//    running maximum by more than 2^8 (the lazy rescale threshold).
#include <type_traits>

#include "pa_internal.cuh"

namespace pa {

namespace {

template <int D, bool FP8>
struct ShortGeom {
    static_assert(!FP8 || D == 128, "the fp8 pool is built for head_dim 128");
    static constexpr int kHalves = FP8 ? 1 : D / 64;          // TMA boxes per 16-key chunk
    static constexpr int kBoxBytes = kChunkKeys * 128;        // 16 rows x 128 B
    static constexpr int kChunkBytes = kHalves * kBoxBytes;   // one 16-key chunk of K (or V)
    // A ring stage holds 32 KB of K and V: 4 chunks (64 keys) of bf16, or 8
    // chunks (128 keys, two of the planner's 64-key stages) of e4m3, so that a
    // consumer warp of an fp8 decode item works on two chunks at once.
    static constexpr int kCPS = FP8 ? 8 : kStageChunks;       // chunks per ring stage
    static constexpr int kPSR = kCPS / kStageChunks;          // planner stages per ring stage
    static constexpr int kRSB = 32 / kCPS;                    // ring stages per block-id batch
    static constexpr int kStageBytes = 2 * kCPS * kChunkBytes;
    static constexpr int kStages = kShortStages;              // ring depth
    // merge scratch (per writer warp): 16 rows x D floats + 16 m + 16 l, kept
    // in the stage being released
    static constexpr int kScratchFloats = 16 * D + 32;
    static constexpr int kCtlBytes = 512;
    static constexpr int kSmemBytes = kStages * kStageBytes + kCtlBytes + 1024;
    static_assert(3 * kScratchFloats * 4 <= kStageBytes, "merge scratch must fit one stage");
};

struct StageMeta {
    int item, stage, flags, pad;
};
// What the consumers need of a work item, handed over by the producer in
// shared memory with the item's first stage (the producer has already
// loaded the record and the request's query start and context), so that an
// item starts without a chain of dependent global loads in the consumers.
struct ItemInfo {
    int b, h, split, nsplit;
    int counter, partial_base, q_begin, q_count;
    int seq_len, stage_end, tok0, ctx;
};
constexpr int kFirst = 1, kLast = 2;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: lazy max update
constexpr int kFoldBatch = 8;              // splits loaded together by the fold
// q is warmed into L2 before the plan completes only when it is this small
// (decode-sized steps); a large step's q mostly feeds the tensor-core kernel
constexpr size_t kPrefetchQMaxBytes = 4u << 20;

__device__ __forceinline__ float quad_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Keep the lower / upper bf16 of a packed pair.
__device__ __forceinline__ uint32_t keep_pair(uint32_t v, bool lo, bool hi) {
    return (lo ? (v & 0xFFFFu) : 0u) | (hi ? (v & 0xFFFF0000u) : 0u);
}

template <int D>
struct Consumer {
    static constexpr int NT = D / 8;   // 8-wide output column tiles
    static constexpr int KS = D / 16;  // 16-deep k steps over the head dim

    // item-wide
    int b, h, tok0, ctx, key_end, R, KQ, rt, kq, nsplit, split, partial_base, counter;
    float sl2, vsc;  // score scale (log2 units) and value scale
    bool swapped;    // fp8 pool, R <= 8: S^T = K Q^T and O^T = V^T P^T
    bool active;
    // per thread: rows g and g+8 of this warp's 16-row tile
    int limit0, limit1;
    uint32_t qa[KS][4];
    float o[NT][4];
    float m0, m1, l0, l1;
};

// Block-table entry of chunk first_stage*4 + lane of a split-KV item -- one
// lane per chunk of an 8-stage batch -- loaded raw; *has = false past the
// item's keys.  The TMA row is computed from it by chunk_row_from, later, so
// that the load's latency overlaps the stages issued in between.  An
// out-of-range table column is clamped and flagged.
__device__ __forceinline__ int chunk_blk_load(const ShortParams &p, const ShortItem &item, int L,
                                              int first_stage, int lane, bool &has) {
    const int key_end = min(item.stage_end * kStageKeys, L);
    const int key0 = (first_stage * kStageChunks + lane) * kChunkKeys;
    has = key0 < key_end;
    if (!has) return 0;
    int col = key0 / p.block_size;
    if (col >= p.bt_stride) {  // seq_len beyond the table row
        flag_status(p.status, PA_DEV_BAD_METADATA);
        col = p.bt_stride - 1;
    }
    return __ldg(p.block_tables + static_cast<int64_t>(item.b) * p.bt_stride + col);
}
// TMA row coordinate (cache row = (block, kv head h, offset)) of that chunk,
// or -1 without one; an out-of-range block id is clamped and flagged.
__device__ __forceinline__ int chunk_row_from(const ShortParams &p, int blk, bool has, int h,
                                              int first_stage, int lane) {
    if (!has) return -1;
    if (blk < 0 || blk >= p.num_blocks) {
        flag_status(p.status, PA_DEV_BAD_BLOCK);
        blk = min(max(blk, 0), p.num_blocks - 1);
    }
    const int key0 = (first_stage * kStageChunks + lane) * kChunkKeys;
    return (blk * p.num_kv_heads + h) * p.block_size + key0 % p.block_size;
}

// L1 prefetch of an item's query rows (q_count tokens x the group's heads,
// each token's group one contiguous run of group * D bf16), by the producer
// lanes right after the item's first stage is issued: the consumers load
// them as mma fragments when that stage lands, and find them in L1.
template <int D>
__device__ __forceinline__ void prefetch_item_q(const ShortParams &p, int tok0, int h,
                                                int q_count, int lane) {
    const int seg = p.group * D * 2;     // bytes of one token's group
    const int lines = (seg + 127) / 128 + 1;  // a run may straddle one more line
    for (int i = lane; i < q_count * lines; i += 32) {
        const int t = i / lines, l = i - t * lines;
        const char *run = reinterpret_cast<const char *>(
            p.q + (static_cast<int64_t>(tok0 + t) * p.num_q_heads + h * p.group) * D);
        const char *a = run + min(l * 128, seg - 1);
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
    }
}

// Work item idx: its record and kv head.
__device__ __forceinline__ ShortItem short_work(const ShortParams &p, int idx, int &h) {
    const int rec = idx / p.num_kv_heads;
    h = idx - rec * p.num_kv_heads;
    return load_record(p.items, rec);
}

// NC (1 or 2) 16-key chunks of an fp8 item with at most 8 rows, operands
// swapped; two chunks are interleaved so their dependency chains overlap.
// Lane (g = lane/4, t = lane%4) holds scores of keys g, g+8 for rows 2t,
// 2t+1, and O^T tile cc's elements (dim 16cc+2g | 16cc+2g+1) x (row 2t |
// 2t+1): cs.o[cc][0] = (row 2t, dim 16cc+2g), [1] = (2t+1, 16cc+2g),
// [2] = (2t, 16cc+2g+1), [3] = (2t+1, 16cc+2g+1).  CHECK = false: every
// key of the chunks is below the item's end and visible to every row (the
// caller checked), so the masks and the V-tail zeroing are compiled out.
template <int D, int NC, bool CHECK>
__device__ __forceinline__ void swapped_chunks(Consumer<D> &cs, const uint32_t (&kb)[NC],
                                               const uint32_t (&vb)[NC], const int (&key0)[NC],
                                               int lane) {
    constexpr int KS = D / 16;
    const int g = lane >> 2, t = lane & 3, mi = lane >> 3;
    // S^T = K Q^T, two accumulators per chunk (even / odd k-steps)
    float st[NC][2][4];
#pragma unroll
    for (int n = 0; n < NC; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) st[n][h][e] = 0.f;
#pragma unroll
    for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
        // matrices: keys 0-7 | 8-15 of k-step 2ks2, then of 2ks2+1
        const int key = (mi & 1) * 8 + (lane & 7);
        const int col = ks2 * 2 + (mi >> 1);
        uint32_t r[NC][4];
#pragma unroll
        for (int n = 0; n < NC; ++n)
            ldsm_x4(kb[n] + sw128_offset(key, col), r[n][0], r[n][1], r[n][2], r[n][3]);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int n = 0; n < NC; ++n) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(r[n][2 * h], a0, a2);      // key g:   dims 4t,4t+1 | 4t+2,4t+3
                e4m3x4_to_f16x2x2(r[n][2 * h + 1], a1, a3);  // key g+8
                const int ks = ks2 * 2 + h;
                mma_f16_16816(st[n][h], a0, a1, a2, a3, cs.qa[ks][0], cs.qa[ks][1]);
            }
    }
    float s[NC][4];
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const bool need_mask =
            CHECK && ((key0[n] + kChunkKeys - 1 > cs.ctx) || (key0[n] + kChunkKeys > cs.key_end));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[n][e] = (st[n][0][e] + st[n][1][e]) * cs.sl2;
            if (need_mask) {
                const int key = key0[n] + g + (e >> 1) * 8;
                const int lim = (e & 1) ? cs.limit1 : cs.limit0;
                if (key > lim || key >= cs.key_end) s[n][e] = -INFINITY;
            }
        }
    }
    // lazy max: reduce over the 8 lanes of a row only when needed
    float la = -INFINITY, lb = -INFINITY;
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        la = fmaxf(la, fmaxf(s[n][0], s[n][2]));
        lb = fmaxf(lb, fmaxf(s[n][1], s[n][3]));
    }
    const bool ua = la > cs.m0 + kRescaleThreshold || (cs.m0 == -INFINITY && la > -INFINITY);
    const bool ub = lb > cs.m1 + kRescaleThreshold || (cs.m1 == -INFINITY && lb > -INFINITY);
    if (__any_sync(0xffffffffu, ua || ub)) {
        float ma = la, mb = lb;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, o));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
        }
        const bool up0 = ma > cs.m0 + kRescaleThreshold || (cs.m0 == -INFINITY && ma > -INFINITY);
        const bool up1 = mb > cs.m1 + kRescaleThreshold || (cs.m1 == -INFINITY && mb > -INFINITY);
        const float a0 = up0 ? (cs.m0 == -INFINITY ? 0.f : fast_exp2(cs.m0 - ma)) : 1.f;
        const float a1 = up1 ? (cs.m1 == -INFINITY ? 0.f : fast_exp2(cs.m1 - mb)) : 1.f;
        if (up0) cs.m0 = ma;
        if (up1) cs.m1 = mb;
        cs.l0 *= a0;
        cs.l1 *= a1;
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) {
            cs.o[cc][0] *= a0;
            cs.o[cc][2] *= a0;
            cs.o[cc][1] *= a1;
            cs.o[cc][3] *= a1;
        }
    }
    const float ref0 = cs.m0 == -INFINITY ? 0.f : cs.m0;
    const float ref1 = cs.m1 == -INFINITY ? 0.f : cs.m1;
    // P^T fragments (key g | g+8) x (rows 2t, 2t+1) -> P fragments of row g
    uint32_t pb0[NC], pb1[NC];
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const float p0 = fast_exp2(s[n][0] - ref0), p1 = fast_exp2(s[n][1] - ref1);
        const float p2 = fast_exp2(s[n][2] - ref0), p3 = fast_exp2(s[n][3] - ref1);
        cs.l0 += p0 + p2;
        cs.l1 += p1 + p3;
        pb0[n] = movmatrix_trans(pack_f16x2(p0, p1));
        pb1[n] = movmatrix_trans(pack_f16x2(p2, p3));
    }
    // O^T += V^T P^T; V rows past the item's keys are zeroed in the fragments
    bool tail[NC], k0[NC], k1[NC], k8[NC], k9[NC];
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const int nvalid = cs.key_end - key0[n];
        tail[n] = CHECK && nvalid < kChunkKeys;
        k0[n] = 2 * t < nvalid;
        k1[n] = 2 * t + 1 < nvalid;
        k8[n] = 2 * t + 8 < nvalid;
        k9[n] = 2 * t + 9 < nvalid;
    }
#pragma unroll
    for (int c2 = 0; c2 < D / 32; ++c2) {
        // matrices: keys 0-7 | 8-15 of dim group 2c2, then of 2c2+1; lane:
        // keys 2t, 2t+1 x dims 2g, 2g+1 of the group
        const int key = (mi & 1) * 8 + (lane & 7);
        const int col = c2 * 2 + (mi >> 1);
        uint32_t r[NC][4];
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            ldsm_x4_t(vb[n] + sw128_offset(key, col), r[n][0], r[n][1], r[n][2], r[n][3]);
            if (tail[n]) {
                r[n][0] = keep_pair(r[n][0], k0[n], k1[n]);
                r[n][2] = keep_pair(r[n][2], k0[n], k1[n]);
                r[n][1] = keep_pair(r[n][1], k8[n], k9[n]);
                r[n][3] = keep_pair(r[n][3], k8[n], k9[n]);
            }
        }
#pragma unroll
        for (int n = 0; n < NC; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t a0, a1, a2, a3;
                // low halves: dim 16cc+2g (A row g), high: 16cc+2g+1 (A row g+8)
                e4m3x4_to_f16x2x2(byte_perm(r[n][2 * h], 0x3120u), a0, a1);
                e4m3x4_to_f16x2x2(byte_perm(r[n][2 * h + 1], 0x3120u), a2, a3);
                mma_f16_16816(cs.o[2 * c2 + h], a0, a1, a2, a3, pb0[n], pb1[n]);
            }
    }
}

// Item epilogue of a swapped fp8 item: row sums over the 8 lanes of a row,
// the 4 consumer warps merged through the stage buffer, then warp 0 writes
// rows 2t and 2t+1 (output, fp32 state for cascade decode, or partial
// state).
template <int D>
__device__ __forceinline__ void swapped_epilogue(Consumer<D> &cs, const ShortParams &p,
                                                 float *scratch, int lane, int warp) {
    constexpr int kRowsFloats = 8 * D;      // floats of one warp's 8 x D block
    constexpr int kSlot = kRowsFloats + 16;  // + 8 maxima + 8 sums
    const int g = lane >> 2, t = lane & 3;
    float la = cs.l0, lb = cs.l1;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, o);
        lb += __shfl_xor_sync(0xffffffffu, lb, o);
    }
    named_bar_sync(1, 32 * kShortConsumerWarps);
    if (cs.kq > 0) {
        float *reg = scratch + (cs.kq - 1) * kSlot;
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) {
            *reinterpret_cast<float2 *>(reg + (2 * t) * D + cc * 16 + 2 * g) =
                make_float2(cs.o[cc][0], cs.o[cc][2]);
            *reinterpret_cast<float2 *>(reg + (2 * t + 1) * D + cc * 16 + 2 * g) =
                make_float2(cs.o[cc][1], cs.o[cc][3]);
        }
        if (g == 0) {
            reg[kRowsFloats + 2 * t] = cs.m0;
            reg[kRowsFloats + 2 * t + 1] = cs.m1;
            reg[kRowsFloats + 8 + 2 * t] = la;
            reg[kRowsFloats + 8 + 2 * t + 1] = lb;
        }
    }
    named_bar_sync(1, 32 * kShortConsumerWarps);
    if (cs.kq != 0) return;
    for (int k = 1; k < cs.KQ; ++k) {
        const float *reg = scratch + (k - 1) * kSlot;
        const float om0 = reg[kRowsFloats + 2 * t], om1 = reg[kRowsFloats + 2 * t + 1];
        const float ol0 = reg[kRowsFloats + 8 + 2 * t], ol1 = reg[kRowsFloats + 8 + 2 * t + 1];
        const float M0 = fmaxf(cs.m0, om0), M1 = fmaxf(cs.m1, om1);
        const float a0 = cs.m0 == -INFINITY ? 0.f : exp2f(cs.m0 - M0);
        const float b0 = om0 == -INFINITY ? 0.f : exp2f(om0 - M0);
        const float a1 = cs.m1 == -INFINITY ? 0.f : exp2f(cs.m1 - M1);
        const float b1 = om1 == -INFINITY ? 0.f : exp2f(om1 - M1);
        la = a0 * la + b0 * ol0;
        lb = a1 * lb + b1 * ol1;
        cs.m0 = M0;
        cs.m1 = M1;
#pragma unroll
        for (int cc = 0; cc < D / 16; ++cc) {
            const float2 x = *reinterpret_cast<const float2 *>(reg + (2 * t) * D + cc * 16 + 2 * g);
            const float2 y = *reinterpret_cast<const float2 *>(reg + (2 * t + 1) * D + cc * 16 + 2 * g);
            cs.o[cc][0] = a0 * cs.o[cc][0] + b0 * x.x;
            cs.o[cc][2] = a0 * cs.o[cc][2] + b0 * x.y;
            cs.o[cc][1] = a1 * cs.o[cc][1] + b1 * y.x;
            cs.o[cc][3] = a1 * cs.o[cc][3] + b1 * y.y;
        }
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = 2 * t + half;
        if (r >= cs.R) continue;
        const float l = half ? lb : la;
        const float m = half ? cs.m1 : cs.m0;
        const float inv = l > 0.f ? cs.vsc / l : 0.f;
        const float lse_v = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        const int tok = cs.tok0 + r / p.group;
        const int hq = cs.h * p.group + r % p.group;
        const int64_t row = static_cast<int64_t>(tok) * p.num_q_heads + hq;
        if (cs.nsplit == 1 && p.out_f32) {
            float *dst = p.out_f32 + row * D;
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc)
                __stcg(reinterpret_cast<float2 *>(dst + cc * 16 + 2 * g),
                       make_float2(cs.o[cc][half] * inv, cs.o[cc][2 + half] * inv));
            if (p.lse && g == 0) p.lse[row] = lse_v;
        } else if (cs.nsplit == 1) {
            uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + row * D);
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc)
                dst[(cc * 16 + 2 * g) >> 1] =
                    pack_bf16x2(cs.o[cc][half] * inv, cs.o[cc][2 + half] * inv);
            if (p.lse && g == 0) p.lse[row] = lse_v;
        } else {
            float *dst = p.partial_o + static_cast<int64_t>(cs.partial_base + r) * D;
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc)
                __stcg(reinterpret_cast<float2 *>(dst + cc * 16 + 2 * g),
                       make_float2(cs.o[cc][half] * inv, cs.o[cc][2 + half] * inv));
            if (g == 0) __stcg(p.partial_lse + cs.partial_base + r, lse_v);
        }
    }
}

}  // namespace

template <int D, bool FP8>
__global__ void __launch_bounds__(kShortThreads, 2)
    short_kernel(const ShortParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
    using G = ShortGeom<D, FP8>;
    constexpr int kStages = G::kStages;
    constexpr int NT = D / 8, KS = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stage_mem = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * G::kStageBytes);
    uint64_t *empty = full + kStages;
    StageMeta *meta = reinterpret_cast<StageMeta *>(empty + kStages);
    int *ctl = reinterpret_cast<int *>(meta + kStages);
    ItemInfo *info = reinterpret_cast<ItemInfo *>(ctl + 16);
    static_assert(kStages * (8 + 8 + 16) + 64 + kStages * sizeof(ItemInfo) <= G::kCtlBytes,
                  "control area");
    volatile int *abort_flag = ctl;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kShortConsumerWarps);
        }
        ctl[0] = 0;
        ctl[1] = 0;
        fence_mbar_init();
    }
    if (warp == kShortConsumerWarps) {
        if (lane == 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
        // Warm L2 with this CTA's slice of the step's metadata (and of q when
        // it is small) while the plan is still running: the first items' block
        // ids and query rows are then L2 hits.  A prefetch is only a hint and
        // reads nothing into registers, so it may run before the wait below.
        const int part = blockIdx.x, parts = gridDim.x;
        l2_prefetch_slice(p.block_tables,
                          static_cast<size_t>(p.num_seqs) * p.bt_stride * sizeof(int), part,
                          parts, lane);
        const size_t q_bytes = static_cast<size_t>(p.num_q_tokens) * p.num_q_heads * D * 2;
        if (q_bytes <= kPrefetchQMaxBytes) l2_prefetch_slice(p.q, q_bytes, part, parts, lane);
        if (part == 0) {
            l2_prefetch_slice(p.qsl, (p.num_seqs + 1) * sizeof(int), 0, 1, lane);
            l2_prefetch_slice(p.ctx, p.num_seqs * sizeof(int), 0, 1, lane);
        }
    }
    __syncthreads();
    // everything below reads the plan's output; after the step's first
    // tensor-core grid (which waited for the plan) there is nothing to wait for
    if (!p.no_start_wait) pdl_wait();
    pdl_trigger();

    auto k_box = [&](int slot, int c, int hf) -> uint8_t * {
        return stage_mem + slot * G::kStageBytes + (c * G::kHalves + hf) * G::kBoxBytes;
    };
    auto v_box = [&](int slot, int c, int hf) -> uint8_t * {
        return stage_mem + slot * G::kStageBytes + G::kCPS * G::kChunkBytes +
               (c * G::kHalves + hf) * G::kBoxBytes;
    };

    const int num_items = *reinterpret_cast<volatile int *>(&p.hdr->num_short_items);

    if (warp == kShortConsumerWarps) {
        // ============================ producer ============================
        uint32_t it = 0;
        bool aborted = false;
        // The next item's index, record, first block ids, query start and
        // context are fetched one dependent step per stage while the current
        // item is still being issued (the steps are taken while the ring is
        // full, or all at the item's last stage), and block ids are read one
        // 8-stage batch ahead, so the ring never waits on a chain of dependent
        // global loads.  When the grid starts at once (it waited for the
        // plan), CTA c starts with item c; beside a tensor-core grid, CTAs
        // start as SMs free up and every item comes from the counter, so the
        // longest items go to the CTAs that start first.
        const int first_static = p.no_start_wait ? 0 : static_cast<int>(gridDim.x);
        int cur_idx = blockIdx.x;
        if (p.no_start_wait) {
            if (lane == 0) cur_idx = atomicAdd(&p.hdr->short_next, 1);
            cur_idx = __shfl_sync(0xffffffffu, cur_idx, 0);
        }
        int cur_h = 0, cur_row = -1, cur_q0 = 0, cur_ctx = 0;
        // the record is loaded together with the item count (records up to
        // max_items exist in the workspace, valid or not)
        ShortItem cur = short_work(p, min(cur_idx, p.max_items - 1), cur_h);
        if (cur_idx < num_items) {
            bool has;
            const int blk = chunk_blk_load(p, cur, cur.seq_len, cur.stage_begin, lane, has);
            cur_q0 = __ldg(p.qsl + cur.b);
            cur_ctx = __ldg(p.ctx + cur.b);
            cur_row = chunk_row_from(p, blk, has, cur_h, cur.stage_begin, lane);
        }
        while (!aborted) {
            if (cur_idx >= num_items) {
                const int slot = it % kStages;
                bool ok = true;
                if (lane == 0) {
                    if (it >= kStages)
                        ok = mbar_wait(&empty[slot], ((it / kStages) - 1) & 1, abort_flag);
                    if (ok) {
                        meta[slot].item = -1;
                        mbar_arrive(&full[slot]);
                    }
                }
                __syncwarp();
                break;
            }
            ShortItem nxt{};
            // prefetch state of the next item
            int nxt_idx = 0, nxt_h = 0, nxt_blk = 0, nxt_q0 = 0, nxt_ctx = 0, pf = 0;
            bool nxt_has = false;
            const int nst = cur.stage_end - cur.stage_begin;  // planner stages
            const int nrs = (nst + G::kPSR - 1) / G::kPSR;     // ring stages
            // The next item is claimed from the counter p.claim_ahead stages
            // before this one ends, so that items go out longest first in the
            // order the CTAs free up (a claim at the item's start would tie a
            // CTA with a long item to a long next item as well); the
            // remaining stages cover the claim's and the prefetch's latency.
            // Beside a mixed step's tensor-core grids the claim is made at
            // the item's start (claim_ahead = 0): there the ragged end of
            // this grid hands SMs to the tensor-core work sooner, measured
            // 1 % faster per step.
            const int rel_claim = p.claim_ahead > 0 ? max(0, nrs - p.claim_ahead) : 0;
            int batch_row = cur_row, next_blk = 0;
            bool next_has = false;
            for (int rel = 0; rel < nrs; ++rel, ++it) {
                const int st = cur.stage_begin + rel * G::kPSR;  // its first planner stage
                if (rel % G::kRSB == 0) {
                    // this batch's rows from the block ids loaded a batch ago;
                    // then the next batch's ids, used only a batch from now
                    if (rel > 0) batch_row = chunk_row_from(p, next_blk, next_has, cur_h, st, lane);
                    next_has = false;
                    if (rel + G::kRSB < nrs)
                        next_blk = chunk_blk_load(p, cur, cur.seq_len, st + 8, lane, next_has);
                }
                if (rel == rel_claim && lane == 0)
                    nxt_idx = atomicAdd(&p.hdr->short_next, 1) + first_static;
                // one prefetch step for the next item per stage after the
                // claim, before this stage's slot is awaited (from the ring's
                // first reuse on); every remaining step at the item's last stage
                for (;;) {
                    if (pf >= 2 || !((it >= kStages && rel > rel_claim) || rel == nrs - 1)) break;
                    if (pf == 0) {
                        nxt_idx = __shfl_sync(0xffffffffu, nxt_idx, 0);
                        nxt = short_work(p, min(nxt_idx, p.max_items - 1), nxt_h);
                        pf = 1;
                    } else {
                        if (nxt_idx < num_items) {
                            nxt_blk = chunk_blk_load(p, nxt, nxt.seq_len, nxt.stage_begin, lane,
                                                     nxt_has);
                            nxt_q0 = __ldg(p.qsl + nxt.b);
                            nxt_ctx = __ldg(p.ctx + nxt.b);
                        }
                        pf = 2;
                    }
                    if (rel != nrs - 1) break;
                }
                // lane c < kCPS takes the row of chunk c of this stage
                const int crow = __shfl_sync(0xffffffffu, batch_row,
                                             (rel % G::kRSB) * G::kCPS + (lane % G::kCPS));
                const int nvalid = __popc(__ballot_sync(0xffffffffu, lane < G::kCPS && crow >= 0));
                const int slot = it % kStages;
                int ok = 1;
                if (lane == 0 && it >= kStages)
                    ok = mbar_wait_spin(&empty[slot], ((it / kStages) - 1) & 1, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                // test hook: stop after the first stage, as a producer would
                // whose wait had run out
                if (p.test_stall && blockIdx.x == 0 && it == 1) ok = 0;
                if (!ok) {
                    aborted = true;
                    break;
                }
                if (lane == 0) {
                    StageMeta mm;
                    mm.item = cur_idx;
                    mm.stage = st;
                    mm.flags = (rel == 0 ? kFirst : 0) | (rel == nrs - 1 ? kLast : 0);
                    mm.pad = 0;
                    meta[slot] = mm;
                    if (rel == 0) {
                        ItemInfo ii;
                        ii.b = cur.b;
                        ii.h = cur_h;
                        ii.split = cur.split;
                        ii.nsplit = cur.nsplit;
                        ii.counter = cur.counter;
                        ii.partial_base = cur.partial_base;
                        ii.q_begin = cur.q_begin;
                        ii.q_count = cur.q_count;
                        ii.seq_len = cur.seq_len;
                        ii.stage_end = cur.stage_end;
                        ii.tok0 = cur_q0;
                        ii.ctx = cur_ctx;
                        info[slot] = ii;
                    }
                    mbar_arrive_expect_tx(&full[slot],
                                          static_cast<uint32_t>(nvalid * 2 * G::kChunkBytes));
                }
                __syncwarp();
                // the stage's chunks' copies are issued by one lane each, at once
                if (lane < G::kCPS && crow >= 0) {
#pragma unroll
                    for (int hf = 0; hf < G::kHalves; ++hf) {
                        tma_load_2d(k_box(slot, lane, hf), &tmk, hf * 64, crow, &full[slot]);
                        tma_load_2d(v_box(slot, lane, hf), &tmv, hf * 64, crow, &full[slot]);
                    }
                }
                if (rel == 0) prefetch_item_q<D>(p, cur_q0 + cur.q_begin, cur_h, cur.q_count, lane);
                __syncwarp();
            }
            if (aborted) break;
            cur_idx = nxt_idx;
            cur = nxt;
            cur_h = nxt_h;
            cur_row = cur_idx < num_items
                          ? chunk_row_from(p, nxt_blk, nxt_has, nxt_h, nxt.stage_begin, lane)
                          : -1;
            cur_q0 = nxt_q0;
            cur_ctx = nxt_ctx;
        }
        if (aborted && lane == 0) {
            flag_status(p.status, PA_DEV_WAIT_TIMEOUT);
            // let copies already in flight land before the CTA exits
            for (uint32_t k = (it > kStages ? it - kStages : 0); k < it; ++k)
                mbar_drain(&full[k % kStages], (k / kStages) & 1);
        }
        return;
    }

    // ============================ consumers ============================
    const int g = lane >> 2, t = lane & 3;
    Consumer<D> cs;
    cs.active = false;
    uint32_t it = 0;
    while (true) {
        const int slot = it % kStages;
        // bf16 consumers poll (they wait on data and leave issue slots to
        // spare); the e4m3 consumers, bound by their own instruction issue,
        // suspend instead (polling measured 1.9 % slower on that mixed step)
        const bool ok = FP8 ? warp_mbar_wait(&full[slot], (it / kStages) & 1, abort_flag)
                            : warp_mbar_wait_spin(&full[slot], (it / kStages) & 1, abort_flag);
        if (!ok) {
            if (lane == 0) flag_status(p.status, PA_DEV_WAIT_TIMEOUT);
            break;
        }
        const StageMeta mm = meta[slot];
        if (mm.item < 0) break;

        if (mm.flags & kFirst) {
            // ---- item setup (the producer's copy of the record) ----
            const ItemInfo item = info[slot];
            const int item_h = item.h;
            cs.b = item.b;
            cs.h = item_h;
            cs.split = item.split;
            cs.nsplit = item.nsplit;
            cs.counter = item.counter * p.num_kv_heads + item_h;
            // a piece of a request: its tokens start q_begin tokens in, so its
            // rows' causal limits start q_begin keys further
            cs.tok0 = item.tok0 + item.q_begin;
            const int n = item.q_count;
            cs.ctx = item.ctx + item.q_begin;
            const int L = item.seq_len;
            cs.key_end = min(item.stage_end * kStageKeys, L);
            cs.R = n * p.group;
            cs.partial_base = item.partial_base + item_h * item.nsplit * cs.R;
            if constexpr (FP8) {
                cs.sl2 = p.scale_log2 * __ldg(p.k_scale + item_h);
                cs.vsc = __ldg(p.v_scale + item_h);
            } else {
                cs.sl2 = p.scale_log2;
                cs.vsc = 1.f;
            }
            const int RT = (cs.R + 15) >> 4;
            const int RTp = RT >= 3 ? 4 : RT;
            cs.KQ = kShortConsumerWarps / RTp;
            cs.rt = warp / cs.KQ;
            cs.kq = warp % cs.KQ;
            cs.active = cs.rt < RT;
            cs.swapped = FP8 && cs.R <= 8;
            const int r0 = cs.rt * 16 + g, r1 = r0 + 8;
            cs.limit0 = r0 < cs.R ? cs.ctx + r0 / p.group : -1;
            cs.limit1 = r1 < cs.R ? cs.ctx + r1 / p.group : -1;
            if (FP8 && cs.swapped) {
                // lane: rows 2t and 2t+1 of the scores, q row g of Q^T; Q^T
                // fragment of k-step ks = q row g, dims 16ks+4t .. +3 (the
                // same dim permutation as the K fragments)
                const int ra = 2 * t, rb = 2 * t + 1;
                cs.limit0 = ra < cs.R ? cs.ctx + ra / p.group : -1;
                cs.limit1 = rb < cs.R ? cs.ctx + rb / p.group : -1;
                const __nv_bfloat16 *qg = nullptr;
                if (g < cs.R)
                    qg = p.q + (static_cast<int64_t>(cs.tok0 + g / p.group) * p.num_q_heads +
                                cs.h * p.group + g % p.group) *
                                   D;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const uint2 x = qg ? __ldg(reinterpret_cast<const uint2 *>(qg) + ks * 4 + t)
                                       : make_uint2(0u, 0u);
                    cs.qa[ks][0] = bf16x2_to_f16x2(x.x);
                    cs.qa[ks][1] = bf16x2_to_f16x2(x.y);
                }
            } else if (cs.active) {
                const __nv_bfloat16 *q0 = nullptr, *q1 = nullptr;
                if (r0 < cs.R)
                    q0 = p.q + (static_cast<int64_t>(cs.tok0 + r0 / p.group) * p.num_q_heads +
                                cs.h * p.group + r0 % p.group) *
                                   D;
                if (r1 < cs.R)
                    q1 = p.q + (static_cast<int64_t>(cs.tok0 + r1 / p.group) * p.num_q_heads +
                                cs.h * p.group + r1 % p.group) *
                                   D;
                if constexpr (FP8) {
                    // k-step ks, lane quad t: dims 16ks+4t .. 16ks+4t+3, as the
                    // fp8 K fragments hold them
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const uint2 z = make_uint2(0u, 0u);
                        const uint2 x0 = q0 ? __ldg(reinterpret_cast<const uint2 *>(q0) + ks * 4 + t) : z;
                        const uint2 x1 = q1 ? __ldg(reinterpret_cast<const uint2 *>(q1) + ks * 4 + t) : z;
                        cs.qa[ks][0] = bf16x2_to_f16x2(x0.x);
                        cs.qa[ks][1] = bf16x2_to_f16x2(x1.x);
                        cs.qa[ks][2] = bf16x2_to_f16x2(x0.y);
                        cs.qa[ks][3] = bf16x2_to_f16x2(x1.y);
                    }
                } else {
                    const uint32_t *w0 = reinterpret_cast<const uint32_t *>(q0);
                    const uint32_t *w1 = reinterpret_cast<const uint32_t *>(q1);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int w = ks * 8 + t;  // 32-bit word index of dims ks*16 + 2t
                        cs.qa[ks][0] = w0 ? __ldg(w0 + w) : 0u;
                        cs.qa[ks][1] = w1 ? __ldg(w1 + w) : 0u;
                        cs.qa[ks][2] = w0 ? __ldg(w0 + w + 4) : 0u;
                        cs.qa[ks][3] = w1 ? __ldg(w1 + w + 4) : 0u;
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) cs.o[nt][e] = 0.f;
            cs.m0 = cs.m1 = -INFINITY;
            cs.l0 = cs.l1 = 0.f;
        }

        // ---- process this warp's chunks of the stage ----
        bool done_swapped = false;
        if constexpr (FP8) {
            if (cs.swapped) {
                // a warp's two chunks of the stage (kq and kq + 4), together
                done_swapped = true;
                const int ka = (mm.stage * kStageChunks + cs.kq) * kChunkKeys;
                const int kb2 = ka + cs.KQ * kChunkKeys;
                if (ka < cs.key_end) {
                    if (kb2 < cs.key_end) {
                        const uint32_t kbs[2] = {smem_u32(k_box(slot, cs.kq, 0)),
                                                 smem_u32(k_box(slot, cs.kq + cs.KQ, 0))};
                        const uint32_t vbs[2] = {smem_u32(v_box(slot, cs.kq, 0)),
                                                 smem_u32(v_box(slot, cs.kq + cs.KQ, 0))};
                        const int ks0[2] = {ka, kb2};
                        // the later chunk's last key decides: below the
                        // item's end and the first row's causal limit, no
                        // key of either chunk needs a mask (one uniform
                        // branch instead of ten per stage)
                        const int last = kb2 + kChunkKeys - 1;
                        if (last < cs.key_end && last <= cs.ctx)
                            swapped_chunks<D, 2, false>(cs, kbs, vbs, ks0, lane);
                        else
                            swapped_chunks<D, 2, true>(cs, kbs, vbs, ks0, lane);
                    } else {
                        const uint32_t kbs[1] = {smem_u32(k_box(slot, cs.kq, 0))};
                        const uint32_t vbs[1] = {smem_u32(v_box(slot, cs.kq, 0))};
                        const int ks0[1] = {ka};
                        swapped_chunks<D, 1, true>(cs, kbs, vbs, ks0, lane);
                    }
                }
            }
        }
        if (cs.active && !done_swapped) {
            for (int c = cs.kq; c < G::kCPS; c += cs.KQ) {
                const int key0 = (mm.stage * kStageChunks + c) * kChunkKeys;
                if (key0 >= cs.key_end) break;
                const uint32_t kb = smem_u32(k_box(slot, c, 0));
                const uint32_t vb = smem_u32(v_box(slot, c, 0));
                const int mi = lane >> 3;
                // The chunk in two compiled forms: CHECK = false when all its
                // keys are below the item's end and visible to every row, so
                // the masks and the V-tail zeroing are compiled out (one
                // uniform branch instead of one per mask and V load group).
                auto chunk = [&](auto check_tag) {
                    constexpr bool CHECK = decltype(check_tag)::value;
                    float sacc[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sacc[i][e] = 0.f;
                    if constexpr (FP8) {
#pragma unroll
                        for (int ks2 = 0; ks2 < KS / 2; ++ks2) {
                            // matrices: keys 0-7 | 8-15 of k-step 2ks2, then of 2ks2+1
                            const int key = (mi & 1) * 8 + (lane & 7);
                            const int col = ks2 * 2 + (mi >> 1);
                            uint32_t r[4];
                            ldsm_x4(kb + sw128_offset(key, col), r[0], r[1], r[2], r[3]);
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const int ks = ks2 * 2 + (m >> 1);
                                uint32_t b0, b1;
                                e4m3x4_to_f16x2x2(r[m], b0, b1);
                                mma_f16_16816(sacc[m & 1], cs.qa[ks][0], cs.qa[ks][1], cs.qa[ks][2],
                                              cs.qa[ks][3], b0, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < KS; ++ks) {
                            const int key = (mi >> 1) * 8 + (lane & 7);
                            const int col = (ks & 3) * 2 + (mi & 1);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(kb + (ks >> 2) * G::kBoxBytes + sw128_offset(key, col), b0, b1,
                                    b2, b3);
                            mma_bf16_16816(sacc[0], cs.qa[ks][0], cs.qa[ks][1], cs.qa[ks][2],
                                           cs.qa[ks][3], b0, b1);
                            mma_bf16_16816(sacc[1], cs.qa[ks][0], cs.qa[ks][1], cs.qa[ks][2],
                                           cs.qa[ks][3], b2, b3);
                        }
                    }
                    // scale to log2 units and mask (causal limit per row, item key range)
                    const bool need_mask = CHECK && ((key0 + kChunkKeys - 1 > cs.ctx) ||
                                                     (key0 + kChunkKeys > cs.key_end));
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float s = sacc[nt][e] * cs.sl2;
                            if (need_mask) {
                                const int key = key0 + nt * 8 + 2 * t + (e & 1);
                                const int lim = (e < 2) ? cs.limit0 : cs.limit1;
                                if (key > lim || key >= cs.key_end) s = -INFINITY;
                            }
                            sacc[nt][e] = s;
                        }
                    float mx0 = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
                    float mx1 = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
                    mx0 = quad_max(mx0);
                    mx1 = quad_max(mx1);
                    const bool up0 = mx0 > cs.m0 + kRescaleThreshold || (cs.m0 == -INFINITY && mx0 > -INFINITY);
                    const bool up1 = mx1 > cs.m1 + kRescaleThreshold || (cs.m1 == -INFINITY && mx1 > -INFINITY);
                    if (__any_sync(0xffffffffu, up0 || up1)) {
                        const float nm0 = up0 ? mx0 : cs.m0;
                        const float nm1 = up1 ? mx1 : cs.m1;
                        const float a0 = up0 ? (cs.m0 == -INFINITY ? 0.f : fast_exp2(cs.m0 - nm0)) : 1.f;
                        const float a1 = up1 ? (cs.m1 == -INFINITY ? 0.f : fast_exp2(cs.m1 - nm1)) : 1.f;
                        cs.m0 = nm0;
                        cs.m1 = nm1;
                        cs.l0 *= a0;
                        cs.l1 *= a1;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            cs.o[nt][0] *= a0;
                            cs.o[nt][1] *= a0;
                            cs.o[nt][2] *= a1;
                            cs.o[nt][3] *= a1;
                        }
                    }
                    const float ref0 = cs.m0 == -INFINITY ? 0.f : cs.m0;
                    const float ref1 = cs.m1 == -INFINITY ? 0.f : cs.m1;
                    float pr[2][4];
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        pr[nt][0] = fast_exp2(sacc[nt][0] - ref0);
                        pr[nt][1] = fast_exp2(sacc[nt][1] - ref0);
                        pr[nt][2] = fast_exp2(sacc[nt][2] - ref1);
                        pr[nt][3] = fast_exp2(sacc[nt][3] - ref1);
                    }
                    cs.l0 += pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
                    cs.l1 += pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
                    const uint32_t pa0 = FP8 ? pack_f16x2(pr[0][0], pr[0][1]) : pack_bf16x2(pr[0][0], pr[0][1]);
                    const uint32_t pa1 = FP8 ? pack_f16x2(pr[0][2], pr[0][3]) : pack_bf16x2(pr[0][2], pr[0][3]);
                    const uint32_t pa2 = FP8 ? pack_f16x2(pr[1][0], pr[1][1]) : pack_bf16x2(pr[1][0], pr[1][1]);
                    const uint32_t pa3 = FP8 ? pack_f16x2(pr[1][2], pr[1][3]) : pack_bf16x2(pr[1][2], pr[1][3]);
                    // V rows past the item's keys may hold anything (even NaN):
                    // zero them in the fragments of a partially valid chunk.
                    const int nvalid = cs.key_end - key0;
                    const bool tail = CHECK && nvalid < kChunkKeys;
                    const bool k0 = 2 * t < nvalid, k1 = 2 * t + 1 < nvalid;
                    const bool k8 = 2 * t + 8 < nvalid, k9 = 2 * t + 9 < nvalid;
                    if constexpr (FP8) {
#pragma unroll
                        for (int c2 = 0; c2 < D / 32; ++c2) {
                            // matrices: keys 0-7 | 8-15 of dim group 2c2, then of 2c2+1;
                            // lane: keys 2t, 2t+1 x dims 2j, 2j+1 (j = lane / 4)
                            const int key = (mi & 1) * 8 + (lane & 7);
                            const int col = c2 * 2 + (mi >> 1);
                            uint32_t r[4];
                            ldsm_x4_t(vb + sw128_offset(key, col), r[0], r[1], r[2], r[3]);
                            if (tail) {
                                r[0] = keep_pair(r[0], k0, k1);
                                r[2] = keep_pair(r[2], k0, k1);
                                r[1] = keep_pair(r[1], k8, k9);
                                r[3] = keep_pair(r[3], k8, k9);
                            }
#pragma unroll
                            for (int m = 0; m < 4; ++m) r[m] = byte_perm(r[m], 0x3120u);
                            // low halves: dim 2j (even tile), high halves: dim 2j+1 (odd tile)
#pragma unroll
                            for (int gsub = 0; gsub < 2; ++gsub) {
                                // keys 0-7 (b0) and 8-15 (b1) of the even and odd tile
                                uint32_t e0, o0, e1, o1;
                                e4m3x4_to_f16x2x2(r[2 * gsub], e0, o0);
                                e4m3x4_to_f16x2x2(r[2 * gsub + 1], e1, o1);
                                mma_f16_16816(cs.o[4 * c2 + 2 * gsub], pa0, pa1, pa2, pa3, e0, e1);
                                mma_f16_16816(cs.o[4 * c2 + 2 * gsub + 1], pa0, pa1, pa2, pa3, o0, o1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int dp = 0; dp < KS; ++dp) {
                            const int key = (mi & 1) * 8 + (lane & 7);
                            const int col = (dp & 3) * 2 + (mi >> 1);
                            uint32_t v0, v1, v2, v3;
                            ldsm_x4_t(vb + (dp >> 2) * G::kBoxBytes + sw128_offset(key, col), v0, v1,
                                      v2, v3);
                            if (tail) {
                                v0 = keep_pair(v0, k0, k1);
                                v2 = keep_pair(v2, k0, k1);
                                v1 = keep_pair(v1, k8, k9);
                                v3 = keep_pair(v3, k8, k9);
                            }
                            mma_bf16_16816(cs.o[2 * dp], pa0, pa1, pa2, pa3, v0, v1);
                            mma_bf16_16816(cs.o[2 * dp + 1], pa0, pa1, pa2, pa3, v2, v3);
                        }
                    }
                };
                if (key0 + kChunkKeys - 1 > cs.ctx || key0 + kChunkKeys > cs.key_end)
                    chunk(std::true_type{});
                else
                    chunk(std::false_type{});
            }
        }

        bool wrote_stage = false;
        if (mm.flags & kLast) {
            // ---- item epilogue ----
            if (FP8 && cs.swapped) {
                swapped_epilogue<D>(cs, p, reinterpret_cast<float *>(stage_mem + slot * G::kStageBytes),
                                    lane, warp);
                wrote_stage = true;
            } else {
                float l0 = quad_sum(cs.l0), l1 = quad_sum(cs.l1);
                if (cs.KQ > 1) {
                    // merge the KQ warps that share a row tile, through this
                    // stage's buffer
                    named_bar_sync(1, 32 * kShortConsumerWarps);
                    float *scratch = reinterpret_cast<float *>(stage_mem + slot * G::kStageBytes);
                    wrote_stage = true;
                    if (cs.active && cs.kq > 0) {
                        float *reg = scratch + (cs.rt * (cs.KQ - 1) + cs.kq - 1) * G::kScratchFloats;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            *reinterpret_cast<float2 *>(reg + g * D + nt * 8 + 2 * t) =
                                make_float2(cs.o[nt][0], cs.o[nt][1]);
                            *reinterpret_cast<float2 *>(reg + (g + 8) * D + nt * 8 + 2 * t) =
                                make_float2(cs.o[nt][2], cs.o[nt][3]);
                        }
                        if (t == 0) {
                            reg[16 * D + g] = cs.m0;
                            reg[16 * D + g + 8] = cs.m1;
                            reg[16 * D + 16 + g] = l0;
                            reg[16 * D + 16 + g + 8] = l1;
                        }
                    }
                    named_bar_sync(1, 32 * kShortConsumerWarps);
                    if (cs.active && cs.kq == 0) {
                        for (int k = 1; k < cs.KQ; ++k) {
                            const float *reg = scratch + (cs.rt * (cs.KQ - 1) + k - 1) * G::kScratchFloats;
                            const float om0 = reg[16 * D + g], om1 = reg[16 * D + g + 8];
                            const float ol0 = reg[16 * D + 16 + g], ol1 = reg[16 * D + 16 + g + 8];
                            const float M0 = fmaxf(cs.m0, om0), M1 = fmaxf(cs.m1, om1);
                            const float a0 = cs.m0 == -INFINITY ? 0.f : exp2f(cs.m0 - M0);
                            const float b0 = om0 == -INFINITY ? 0.f : exp2f(om0 - M0);
                            const float a1 = cs.m1 == -INFINITY ? 0.f : exp2f(cs.m1 - M1);
                            const float b1 = om1 == -INFINITY ? 0.f : exp2f(om1 - M1);
                            l0 = a0 * l0 + b0 * ol0;
                            l1 = a1 * l1 + b1 * ol1;
                            cs.m0 = M0;
                            cs.m1 = M1;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const float2 x = *reinterpret_cast<const float2 *>(reg + g * D + nt * 8 + 2 * t);
                                const float2 y = *reinterpret_cast<const float2 *>(reg + (g + 8) * D + nt * 8 + 2 * t);
                                cs.o[nt][0] = a0 * cs.o[nt][0] + b0 * x.x;
                                cs.o[nt][1] = a0 * cs.o[nt][1] + b0 * x.y;
                                cs.o[nt][2] = a1 * cs.o[nt][2] + b1 * y.x;
                                cs.o[nt][3] = a1 * cs.o[nt][3] + b1 * y.y;
                            }
                        }
                    }
                }
                if (cs.active && cs.kq == 0) {
                    // final state of rows r0 = rt*16+g and r1 = r0+8 over this item's keys.
                    // Output columns in pairs: pair pi of this lane holds dims
                    // (col, col+1) -- bf16 ring: tile pi; fp8 ring: the even and
                    // odd tiles of dim group pi/2 (see the header comment)
                    auto pair_of = [&](int pi, int half, float &x, float &y) -> int {
                        if constexpr (FP8) {
                            const int grp = pi >> 1, e = pi & 1;
                            x = cs.o[2 * grp][2 * half + e];
                            y = cs.o[2 * grp + 1][2 * half + e];
                            return grp * 16 + 4 * t + 2 * e;
                        } else {
                            x = cs.o[pi][2 * half];
                            y = cs.o[pi][2 * half + 1];
                            return pi * 8 + 2 * t;
                        }
                    };
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int r = cs.rt * 16 + g + half * 8;
                        if (r >= cs.R) continue;
                        const float l = half ? l1 : l0;
                        const float m = half ? cs.m1 : cs.m0;
                        const float inv = l > 0.f ? cs.vsc / l : 0.f;
                        const float lse_v = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
                        const int tok = cs.tok0 + r / p.group;
                        const int hq = cs.h * p.group + r % p.group;
                        const int64_t row = static_cast<int64_t>(tok) * p.num_q_heads + hq;
                        if (cs.nsplit == 1) {
                            if (p.out_f32) {
                                float *dst = p.out_f32 + row * D;
#pragma unroll
                                for (int pi = 0; pi < NT; ++pi) {
                                    float x, y;
                                    const int col = pair_of(pi, half, x, y);
                                    __stcg(reinterpret_cast<float2 *>(dst + col),
                                           make_float2(x * inv, y * inv));
                                }
                            } else {
                                uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + row * D);
#pragma unroll
                                for (int pi = 0; pi < NT; ++pi) {
                                    float x, y;
                                    const int col = pair_of(pi, half, x, y);
                                    dst[col >> 1] = pack_bf16x2(x * inv, y * inv);
                                }
                            }
                            if (p.lse && t == 0) p.lse[row] = lse_v;
                        } else {
                            float *dst = p.partial_o + static_cast<int64_t>(cs.partial_base + r) * D;
#pragma unroll
                            for (int pi = 0; pi < NT; ++pi) {
                                float x, y;
                                const int col = pair_of(pi, half, x, y);
                                __stcg(reinterpret_cast<float2 *>(dst + col), make_float2(x * inv, y * inv));
                            }
                            if (t == 0) __stcg(p.partial_lse + cs.partial_base + r, lse_v);
                        }
                    }
                }
            }
            if (cs.nsplit > 1) {
                // fused split-KV epilogue: the last split of (b, h) folds all
                // partials.  One thread's acquire-release counter update
                // releases this CTA's partial writes (ordered before it by the
                // CTA barrier) and, if it is the last, acquires the others'.
                named_bar_sync(1, 32 * kShortConsumerWarps);
                if (threadIdx.x == 0)
                    ctl[1] = atomic_add_acq_rel_gpu(p.counters + cs.counter, 1) == cs.nsplit - 1;
                named_bar_sync(1, 32 * kShortConsumerWarps);
                if (*reinterpret_cast<volatile int *>(&ctl[1])) {
                    const int base = cs.partial_base - cs.split * cs.R;
                    const int total4 = cs.R * (D / 4);
                    for (int idx = threadIdx.x; idx < total4; idx += 32 * kShortConsumerWarps) {
                        const int r = idx / (D / 4), e4 = idx - r * (D / 4);
                        const int tok = cs.tok0 + r / p.group;
                        const int hq = cs.h * p.group + r % p.group;
                        const int64_t row = static_cast<int64_t>(tok) * p.num_q_heads + hq;
                        const float *pl = p.partial_lse + base + r;
                        const float4 *po = reinterpret_cast<const float4 *>(
                                               p.partial_o + static_cast<int64_t>(base + r) * D) + e4;
                        const int64_t ostride = static_cast<int64_t>(cs.R) * (D / 4);
                        // splits are read kFoldBatch at a time so their L2
                        // round trips overlap
                        float M = -INFINITY;
                        for (int s0 = 0; s0 < cs.nsplit; s0 += kFoldBatch) {
#pragma unroll
                            for (int j = 0; j < kFoldBatch; ++j)
                                if (s0 + j < cs.nsplit) M = fmaxf(M, __ldcg(pl + (s0 + j) * cs.R));
                        }
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        float wsum = 0.f;
                        if (M != -INFINITY) {
                            for (int s0 = 0; s0 < cs.nsplit; s0 += kFoldBatch) {
                                float lv[kFoldBatch];
                                float4 v[kFoldBatch];
#pragma unroll
                                for (int j = 0; j < kFoldBatch; ++j) {
                                    const bool in = s0 + j < cs.nsplit;
                                    lv[j] = in ? __ldcg(pl + (s0 + j) * cs.R) : -INFINITY;
                                    v[j] = in ? __ldcg(po + (s0 + j) * ostride)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                                }
#pragma unroll
                                for (int j = 0; j < kFoldBatch; ++j) {
                                    const float w = __expf(lv[j] - M);
                                    wsum += w;
                                    acc.x += w * v[j].x;
                                    acc.y += w * v[j].y;
                                    acc.z += w * v[j].z;
                                    acc.w += w * v[j].w;
                                }
                            }
                        }
                        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
                        if (p.out_f32) {
                            __stcg(reinterpret_cast<float4 *>(p.out_f32 + row * D) + e4,
                                   make_float4(acc.x * inv, acc.y * inv, acc.z * inv,
                                               acc.w * inv));
                        } else {
                            uint2 pk2;
                            pk2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                            pk2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                            reinterpret_cast<uint2 *>(p.out + row * D)[e4] = pk2;
                        }
                        if (e4 == 0 && p.lse) p.lse[row] = wsum > 0.f ? M + __logf(wsum) : -INFINITY;
                    }
                }
                named_bar_sync(1, 32 * kShortConsumerWarps);
            }
        }
        if (wrote_stage) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        ++it;
    }
}

size_t short_smem_bytes(int head_dim) {
    return head_dim == 128 ? ShortGeom<128, false>::kSmemBytes : ShortGeom<64, false>::kSmemBytes;
}

template <int D, bool FP8>
static int configure_short() {
    static PerDeviceOnce once;
    return once_per_device(once, [] {
        return cudaFuncSetAttribute(short_kernel<D, FP8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    ShortGeom<D, FP8>::kSmemBytes);
    });
}

template <int D, bool FP8>
static int max_ctas() {
    int n = 0;
    if (configure_short<D, FP8>() != PA_OK) return 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, short_kernel<D, FP8>, kShortThreads,
                                                  ShortGeom<D, FP8>::kSmemBytes);
    return n > 0 ? n : 1;
}

int short_max_ctas_per_sm(int head_dim, bool fp8) {
    if (fp8) return max_ctas<128, true>();
    return head_dim == 128 ? max_ctas<128, false>() : max_ctas<64, false>();
}

template <int D, bool FP8>
static int launch(const ShortParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int grid,
                  cudaStream_t s) {
    if (configure_short<D, FP8>() != PA_OK) return PA_ERR_CUDA;
    PdlLaunch l(grid, kShortThreads, ShortGeom<D, FP8>::kSmemBytes, s);
    return launch_kernel(l, short_kernel<D, FP8>, p, tk, tv) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int launch_short(const ShortParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                 int head_dim, bool fp8, int grid, cudaStream_t s) {
    if (grid <= 0) return PA_OK;
    if (fp8) return head_dim == 128 ? launch<128, true>(p, tk, tv, grid, s) : PA_ERR_UNSUPPORTED;
    return head_dim == 128 ? launch<128, false>(p, tk, tv, grid, s)
                           : launch<64, false>(p, tk, tv, grid, s);
}

}  // namespace pa
