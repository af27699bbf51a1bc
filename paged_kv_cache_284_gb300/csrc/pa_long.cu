// pa_long.cu -- tensor-core attention for long query rows: chunked-prefill
// chunks, prefix-cache hits and whole prompts ("vLLM中如何实现大模型推理加速
// 技术？": chunked prefill / prefix caching; "11. 推理加速(一):vLLM 原理",
// §11.3: prefill is compute-bound), and the cascade shared-prefix pass
// (2048ai.net page on the vLLM V1 engine, §02.1 级联推理: one multi-query
// pass over the shared KV, each prefix block read once per 128 query rows).
//
// One CTA computes a 128-row query tile against a key range, FlashAttention
// style, on the 5th-generation tensor cores:
//  * rows of the tile are (token, head) pairs of one kv head's GQA group:
//    128 / group tokens x group heads, loaded by one 3-D TMA box per 64 dims;
//  * K and V tiles of 128 keys are gathered through the block table as eight
//    16-key TMA boxes (128-byte swizzle) into a 2-deep ring;
//  * warp 1 issues tcgen05.mma: S = Q K^T (M=128, N=128, K=head_dim) into one
//    of two TMEM S buffers, then O += P V (M=128, N=head_dim, K=128) into a
//    TMEM O accumulator, V read N-major straight from its cache layout;
//  * warps 2-5 (one thread per row) read S from TMEM, apply the
//    context-offset causal mask (row i of a request with context c sees keys
//    0..c+i), run the online softmax in the log2 domain with a lazy max
//    update, rescale O in TMEM only when the max grows by more than 2^8, and
//    write P (bf16) to shared memory for the next MMA;
//  * the epilogue reads O from TMEM, normalises and stores bf16 (or fp32
//    partial states that the last split folds with the merge operator).
// Key tiles entirely above a tile's causal limit are never visited.
#include "pa_internal.cuh"

namespace pa {

namespace {

template <int D>
struct LongGeom {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = 128 * 128;            // 128 rows x 128 B
    static constexpr int kQBytes = kHalves * kHalfBytes;    // Q tile
    static constexpr int kKVBytes = kHalves * kHalfBytes;   // one K (or V) tile of 128 keys
    static constexpr int kPBytes = 2 * kHalfBytes;          // P tile: 128 rows x 128 keys
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + 2 * kKVBytes;
    static constexpr int kOffP = kOffV + 2 * kKVBytes;
    static constexpr int kOffBar = kOffP + kPBytes;
    static constexpr int kCtlBytes = 256;
    // at least 116 KiB so that one CTA owns an SM (and its 512 TMEM columns)
    static constexpr int kSmemRaw = kOffBar + kCtlBytes + 1024;
    static constexpr int kSmemBytes = kSmemRaw > 116 * 1024 ? kSmemRaw : 116 * 1024;
    static constexpr uint32_t kTmemCols = 512;  // S0 | S1 | O
    static constexpr int kColS = 0, kColO = 2 * kLongKeys;
};

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;

struct Bars {
    uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full, o_done, sync, drain;
};

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Barrier among the 4 softmax warps built on an mbarrier with a bounded
// wait, so a kernel that gave up elsewhere can never hang here.
__device__ __forceinline__ bool softmax_sync(uint64_t *bar, uint32_t &phase, volatile int *abort) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = warp_wait(bar, phase & 1, abort);
    ++phase;
    return ok;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kLongThreads, 1)
    long_kernel(const LongParams p, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using G = LongGeom<D>;
    constexpr int KS = D / 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars *bars = reinterpret_cast<Bars *>(smem + G::kOffBar);
    int *ctl = reinterpret_cast<int *>(smem + G::kOffBar + 128);
    volatile int *abort_flag = ctl;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctl + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- item ---------------------------------------------------------------
    int b = 0, h, tok0, nvalid, pos0, key_begin, key_end, causal, nsplit = 1, split = 0;
    int counter_idx = 0, partial_base = 0;
    const int TQ = p.q_tile_tokens;
    if (!p.prefix_mode) {
        const int num_items = *reinterpret_cast<volatile int *>(&p.hdr->num_long_items);
        if (static_cast<int>(blockIdx.x) >= num_items) return;
        const LongItem it = p.items[blockIdx.x];
        b = it.b;
        h = it.h;
        const int q0 = __ldg(p.qsl + b);
        const int n = __ldg(p.qsl + b + 1) - q0;
        tok0 = q0 + it.q_tile * TQ;
        nvalid = min(TQ, n - it.q_tile * TQ);
        pos0 = __ldg(p.ctx + b) + it.q_tile * TQ;
        key_begin = it.key_begin;
        key_end = it.key_end;
        causal = 1;
    } else {
        const int total = p.num_kv_heads * p.prefix_q_tiles * p.prefix_nsplit;
        if (static_cast<int>(blockIdx.x) >= total) return;
        const int idx = blockIdx.x;
        split = idx % p.prefix_nsplit;
        const int qt = (idx / p.prefix_nsplit) % p.prefix_q_tiles;
        h = idx / (p.prefix_nsplit * p.prefix_q_tiles);
        nsplit = p.prefix_nsplit;
        tok0 = qt * TQ;
        nvalid = min(TQ, p.num_q_tokens - tok0);
        pos0 = 0;
        key_begin = split * p.prefix_split_keys;
        key_end = min(p.prefix_len, key_begin + p.prefix_split_keys);
        causal = 0;
        counter_idx = h * p.prefix_q_tiles + qt;
        partial_base = counter_idx * nsplit * kLongRows;
    }
    const int span = key_end - key_begin;
    const int nt = span > 0 ? (span + kLongKeys - 1) / kLongKeys : 0;
    const int *bt = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;

    // ---- setup ----------------------------------------------------------------
    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->kv_full[i], 1);
            mbar_init(&bars->kv_empty[i], 1);
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], 4);
        }
        mbar_init(&bars->p_full, 4);
        mbar_init(&bars->o_done, 1);
        mbar_init(&bars->sync, 4);
        mbar_init(&bars->drain, 1);
        ctl[0] = 0;
        ctl[1] = 0;
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
    uint8_t *sP = smem + G::kOffP;

    if (warp == 0) {
        // ============================ producer ============================
        int issued = 0;
        if (nt > 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tmq);
                tma_prefetch_desc(&tmk);
                tma_prefetch_desc(&tmv);
                mbar_arrive_expect_tx(&bars->q_full,
                                      static_cast<uint32_t>(G::kHalves * 128 * p.group * TQ));
                for (int hf = 0; hf < G::kHalves; ++hf)
                    tma_load_3d(sQ + hf * G::kHalfBytes, &tmq, hf * 64, h * p.group, tok0,
                                &bars->q_full);
            }
            int my_row = p.kv_rows;
            for (int j = 0; j < nt; ++j) {
                const int st = j & 1;
                if ((j & 3) == 0) {
                    // rows of the next 32 chunks (4 tiles), one per lane;
                    // chunks past key_end read fully out of bounds -> zeros
                    const int key0 = key_begin + (j * 8 + lane) * kChunkKeys;
                    my_row = p.kv_rows;
                    if (key0 < key_end) {
                        int col = key0 / p.block_size;
                        if (p.bt_stride > 0 && col >= p.bt_stride) {  // beyond the table row
                            flag_status(p.status, PA_DEV_BAD_METADATA);
                            col = p.bt_stride - 1;
                        }
                        int blk = __ldg(bt + col);
                        if (blk < 0 || blk >= p.num_blocks) {
                            flag_status(p.status, PA_DEV_BAD_BLOCK);
                            blk = min(max(blk, 0), p.num_blocks - 1);
                        }
                        my_row = (blk * p.num_kv_heads + h) * p.block_size + key0 % p.block_size;
                    }
                }
                if (j >= 2 && !warp_wait(&bars->kv_empty[st], ((j - 2) >> 1) & 1, abort_flag))
                    break;
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars->kv_full[st],
                                          static_cast<uint32_t>(2 * G::kKVBytes));
                __syncwarp();
                const int c = lane & 7;
                const int row = __shfl_sync(0xffffffffu, my_row, (j & 3) * 8 + c);
                if (lane < 8) {
                    for (int hf = 0; hf < G::kHalves; ++hf) {
                        tma_load_2d(sK + st * G::kKVBytes + hf * G::kHalfBytes + c * 2048, &tmk,
                                    hf * 64, row, &bars->kv_full[st]);
                        tma_load_2d(sV + st * G::kKVBytes + hf * G::kHalfBytes + c * 2048, &tmv,
                                    hf * 64, row, &bars->kv_full[st]);
                    }
                }
                __syncwarp();
                issued = j + 1;
            }
        }
        if (*abort_flag && lane == 0) {
            for (int j = max(0, issued - 2); j < issued; ++j)
                mbar_drain(&bars->kv_full[j & 1], (j >> 1) & 1);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0 && nt > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kLongRows, kLongKeys, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kLongRows, D, 1);
            const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV),
                           p_addr = smem_u32(sP);
            bool ok = mbar_wait(&bars->q_full, 0, abort_flag);
            auto issue_pv = [&](int i) -> bool {
                if (!mbar_wait(&bars->p_full, i & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t vs = v_addr + (i & 1) * G::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kLongKeys / 16; ++kk) {
                    const uint64_t ad = smem_desc_sw128(
                        p_addr + (kk >> 2) * G::kHalfBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(vs + kk * 2048, G::kHalfBytes, 1024);
                    tc_mma(tmem + G::kColO, ad, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars->kv_empty[i & 1]);
                tc_commit(&bars->o_done);
                return true;
            };
            for (int j = 0; ok && j < nt; ++j) {
                const int st = j & 1;
                if (!mbar_wait(&bars->kv_full[st], (j >> 1) & 1, abort_flag)) { ok = false; break; }
                if (j >= 2 && !mbar_wait(&bars->s_free[st], ((j - 2) >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ks = k_addr + st * G::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint64_t ad = smem_desc_sw128(
                        q_addr + (kk >> 2) * G::kHalfBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(
                        ks + (kk >> 2) * G::kHalfBytes + (kk & 3) * 32, 16, 1024);
                    tc_mma(tmem + G::kColS + st * kLongKeys, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars->s_full[st]);
                if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) ok = issue_pv(nt - 1);
            if (!ok) {
                // let every MMA already issued finish before TMEM is released
                tc_commit(&bars->drain);
                mbar_drain(&bars->drain, 0);
            }
        }
    } else {
        // ============================ softmax + epilogue ============================
        const int wq = warp & 3;  // TMEM lane quarter of this warp
        const int r = wq * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const int ttok = r / p.group;
        const int jh = r - ttok * p.group;
        const bool row_valid = ttok < nvalid && r < TQ * p.group;
        const int row_limit = causal ? pos0 + ttok : 0x7fffffff;
        const int tile_limit_min = causal ? pos0 : 0x7fffffff;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int sb = j & 1;
            if (!warp_wait(&bars->s_full[sb], (j >> 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            float s[kLongKeys];
            {
                uint32_t raw[32];
#pragma unroll
                for (int qd = 0; qd < kLongKeys / 32; ++qd) {
                    tmem_ld32(t_lane + G::kColS + sb * kLongKeys + qd * 32, raw);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[qd * 32 + i] = __uint_as_float(raw[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free[sb]);
            const int kb = key_begin + j * kLongKeys;
            const bool need_mask = (kb + kLongKeys - 1 > tile_limit_min) || (kb + kLongKeys > key_end);
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kLongKeys; ++i) {
                float v = s[i] * p.scale_log2;
                if (need_mask && (kb + i > row_limit || kb + i >= key_end)) v = -INFINITY;
                s[i] = v;
                mx = fmaxf(mx, v);
            }
            const bool up = mx > m_used + kRescaleThreshold || (m_used == -INFINITY && mx > -INFINITY);
            float alpha = 1.f;
            if (up) {
                alpha = m_used == -INFINITY ? 0.f : exp2f(m_used - mx);
                m_used = mx;
            }
            const float ref = m_used == -INFINITY ? 0.f : m_used;
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < kLongKeys; ++i) {
                s[i] = exp2f(s[i] - ref);
                sum += s[i];
            }
            l = l * alpha + sum;
            if (j >= 1) {
                if (!warp_wait(&bars->o_done, (j - 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    uint32_t raw[32];
#pragma unroll
                    for (int qd = 0; qd < D / 32; ++qd) {
                        tmem_ld32(t_lane + G::kColO + qd * 32, raw);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
                        tmem_st32(t_lane + G::kColO + qd * 32, raw);
                    }
                    tmem_wait_st();
                }
            }
            if (kb + kLongKeys > key_end) {
                // the last loaded chunk may extend past the keys: zero those V
                // rows so 0-probabilities never meet non-finite cache contents
                if (!warp_wait(&bars->kv_full[sb], (j >> 1) & 1, abort_flag)) { ok = false; break; }
                const int z0 = key_end - kb;                     // first row to clear
                const int z1 = min(kLongKeys, (z0 + 15) & ~15);  // end of its chunk
                const int pieces = (z1 - z0) * 8 * G::kHalves;   // 16-byte pieces
                for (int idx = r; idx < pieces; idx += 128) {
                    const int hf = idx / ((z1 - z0) * 8);
                    const int rem = idx - hf * (z1 - z0) * 8;
                    const int row = z0 + rem / 8, piece = rem % 8;
                    *reinterpret_cast<uint4 *>(sV + sb * G::kKVBytes + hf * G::kHalfBytes +
                                               row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            // P row r (bf16) into the K-major, 128-byte swizzled A-operand tile
#pragma unroll
            for (int c16 = 0; c16 < kLongKeys / 8; ++c16) {
                uint4 v;
                v.x = pack_bf16x2(s[c16 * 8 + 0], s[c16 * 8 + 1]);
                v.y = pack_bf16x2(s[c16 * 8 + 2], s[c16 * 8 + 3]);
                v.z = pack_bf16x2(s[c16 * 8 + 4], s[c16 * 8 + 5]);
                v.w = pack_bf16x2(s[c16 * 8 + 6], s[c16 * 8 + 7]);
                *reinterpret_cast<uint4 *>(sP + (c16 >> 3) * G::kHalfBytes +
                                           sw128_offset(r, c16 & 7)) = v;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full);
        }
        if (ok && nt > 0) ok = warp_wait(&bars->o_done, (nt - 1) & 1, abort_flag);
        tc_fence_after();

        // ---- epilogue ----
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse_v = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
        const int tok = tok0 + ttok;
        const int hq = h * p.group + jh;
        const int64_t orow = static_cast<int64_t>(tok) * p.num_q_heads + hq;
        const bool direct = nsplit == 1;
        const int64_t prow = static_cast<int64_t>(partial_base + split * kLongRows + r);
        for (int qd = 0; qd < D / 32; ++qd) {
            uint32_t raw[32];
            if (ok && nt > 0) {
                tmem_ld32(t_lane + G::kColO + qd * 32, raw);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) raw[i] = 0u;
            }
            if (!ok || !row_valid) continue;
            if (direct && !p.out_f32) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + qd * 32);
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
                float *dst = direct ? p.out_f32 + orow * D + qd * 32 : p.partial_o + prow * D + qd * 32;
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                    __stcg(reinterpret_cast<float4 *>(dst) + v4,
                           make_float4(__uint_as_float(raw[v4 * 4 + 0]) * inv, __uint_as_float(raw[v4 * 4 + 1]) * inv,
                                       __uint_as_float(raw[v4 * 4 + 2]) * inv, __uint_as_float(raw[v4 * 4 + 3]) * inv));
            }
        }
        if (ok && row_valid) {
            if (direct) {
                if (p.lse) p.lse[orow] = lse_v;
            } else {
                __stcg(p.partial_lse + prow, lse_v);
            }
        }
        if (!direct) {
            // fused split epilogue: the last split of this (kv head, query tile)
            // folds the partial states with the merge operator
            uint32_t phase = 0;
            __threadfence();
            bool sok = softmax_sync(&bars->sync, phase, abort_flag);
            if (sok && r == 0) {
                const int old = atomicAdd(p.counters + counter_idx, 1);
                ctl[1] = (old == nsplit - 1) ? 1 : 0;
            }
            sok = softmax_sync(&bars->sync, phase, abort_flag) && sok;
            if (sok && ctl[1] && row_valid) {
                __threadfence();
                const int64_t base = partial_base + r;
                float M = -INFINITY;
                for (int s2 = 0; s2 < nsplit; ++s2)
                    M = fmaxf(M, __ldcg(p.partial_lse + base + s2 * kLongRows));
                float wsum = 0.f;
                float w[64];
                const int ns = min(nsplit, 64);
                for (int s2 = 0; s2 < ns; ++s2) {
                    const float ls = __ldcg(p.partial_lse + base + s2 * kLongRows);
                    w[s2] = M == -INFINITY ? 0.f : __expf(ls - M);
                    wsum += w[s2];
                }
                const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
                for (int e4 = 0; e4 < D / 4; ++e4) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int s2 = 0; s2 < ns; ++s2) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                                    p.partial_o + (base + s2 * kLongRows) * D) + e4);
                        acc.x += w[s2] * v.x;
                        acc.y += w[s2] * v.y;
                        acc.z += w[s2] * v.z;
                        acc.w += w[s2] * v.w;
                    }
                    acc.x *= winv;
                    acc.y *= winv;
                    acc.z *= winv;
                    acc.w *= winv;
                    if (p.out_f32) {
                        reinterpret_cast<float4 *>(p.out_f32 + orow * D)[e4] = acc;
                    } else {
                        uint2 pk;
                        pk.x = pack_bf16x2(acc.x, acc.y);
                        pk.y = pack_bf16x2(acc.z, acc.w);
                        reinterpret_cast<uint2 *>(p.out + orow * D)[e4] = pk;
                    }
                }
                if (p.lse) p.lse[orow] = wsum > 0.f ? M + __logf(wsum) : -INFINITY;
            }
        }
    }

    if (*abort_flag && threadIdx.x == 0) flag_status(p.status, PA_DEV_WAIT_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, G::kTmemCols);
}

size_t long_smem_bytes(int head_dim) {
    return head_dim == 128 ? LongGeom<128>::kSmemBytes : LongGeom<64>::kSmemBytes;
}

template <int D>
static int configure_long() {
    static bool done = false;
    if (!done) {
        if (cudaFuncSetAttribute(long_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 LongGeom<D>::kSmemBytes) != cudaSuccess)
            return PA_ERR_CUDA;
        done = true;
    }
    return PA_OK;
}

int launch_long(const LongParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                const CUtensorMap &tv, int head_dim, int grid, cudaStream_t s) {
    if (grid <= 0) return PA_OK;
    if (head_dim == 128) {
        if (configure_long<128>() != PA_OK) return PA_ERR_CUDA;
        long_kernel<128><<<grid, kLongThreads, LongGeom<128>::kSmemBytes, s>>>(p, tq, tk, tv);
    } else {
        if (configure_long<64>() != PA_OK) return PA_ERR_CUDA;
        long_kernel<64><<<grid, kLongThreads, LongGeom<64>::kSmemBytes, s>>>(p, tq, tk, tv);
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
