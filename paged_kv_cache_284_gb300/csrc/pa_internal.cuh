// pa_internal.cuh -- shared device helpers and plan structures of libpa.
//
// Inline-PTX wrappers for the sm_100-family async machinery the kernels use:
// mbarriers with bounded waits, TMA tensor loads (cp.async.bulk.tensor),
// tcgen05 MMA / TMEM, and the warp-level mma.sync used by the memory-bound
// split-KV kernel.  Nothing here computes attention; the kernels do.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "../../include/pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// Geometry shared by host planner and kernels
// ---------------------------------------------------------------------------
constexpr int kChunkKeys = 16;        // keys per TMA box (rows of one cache box)
constexpr int kStageChunks = 4;       // split-KV kernel: chunks per pipeline stage
constexpr int kStageKeys = kChunkKeys * kStageChunks;  // 64 keys per stage
constexpr int kShortStages = 3;       // split-KV kernel: pipeline depth
constexpr int kShortMaxRows = 64;     // rows (q_len * group) a split-KV item may hold
constexpr int kShortConsumerWarps = 4;
constexpr int kShortThreads = 32 * (kShortConsumerWarps + 1);
constexpr int kLongRows = 128;        // tcgen05 tile: M = 128 query rows
constexpr int kLongKeys = 128;        // tcgen05 tile: N = 128 keys per KV tile
constexpr int kLongThreads = 384;     // 12 warps: K+Q loads, QK^T, 8 x softmax, V loads, PV
constexpr int kPlanThreads = 1024;
constexpr int kSmallPlanSeqs = 16;    // steps of at most this many requests plan on one warp
constexpr int kMinSplitStages = 4;    // 256 keys: smallest automatic split
// Automatic split size: total split-KV stages / (this x persistent CTAs).  The
// items are taken longest first, so a request is cut only when it is long
// next to a CTA's share of the step (each split costs a partial-state write
// and a fold).
constexpr int kSplitItemsPerCta = 3;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s per pipeline wait
// split-KV kernel: a CTA claims its next work item this many ring stages
// before its current one ends (enough to hide the claim and the prefetch of
// the item's record and first block ids).  Measured per call: cascade 63.7 /
// 63.3 / 63.0 / 65.7 / 66.4 us with 2 / 3 / 4 / 6 / 8 stages; decode-heavy
// and 64-request decode steps best or tied at 4.
constexpr int kClaimAheadStages = 4;

// Work list written by the plan kernel into the caller's workspace.
struct PlanHeader {
    int num_short_items;   // work items (records x Hkv)
    int num_long_items;    // work items (records x Hkv)
    int short_next;        // dynamic work counter of the split-KV kernel
    int long_next;         // dynamic work counter of the tensor-core kernel
    int split_stages;      // chosen split size (in 64-key stages)
    int partial_rows;      // partial-state rows used
    int num_staged;        // fp8 pool: long requests given a bf16 staging copy
    int staged_blocks;     // staging blocks used
    int first_done;        // CTAs of the first tensor-core launch that finished
    int pad[7];
};
static_assert(sizeof(PlanHeader) == 64, "header size");

// Work records written by the plan kernel.  A record covers every kv head:
// work item i of a kernel is record i / Hkv for kv head i % Hkv, so the plan
// writes one 32-byte record (two 16-byte stores) per request split or query
// tile instead of one per kv head.

// Split-KV record: query tokens [q_begin, q_begin + q_count) of request b
// (a whole short request, or one piece of a longer one), keys
// [stage_begin*64, min(stage_end*64, seq_len)).  Split s of kv head h writes
// partial rows partial_base + h*nsplit*R + [0, R) (R = q_count * group) when
// nsplit > 1, and counts its completion in counters[counter*Hkv + h].
struct alignas(16) ShortItem {
    int b, split, nsplit, stage_begin;
    int stage_end, partial_base, q_begin, q_count;
    int counter, seq_len, pad1, pad2;  // seq_len: the request's, read once by the plan
};
static_assert(sizeof(ShortItem) == 48, "item size");

// Tensor-core record: query tile q_tile of request b (tile = 128/group tokens
// x group heads), keys [key_begin, key_end).
struct alignas(16) LongItem {
    int b, q_tile, key_begin, key_end;
    int pad[4];
};
static_assert(sizeof(LongItem) == 32, "item size");

#if defined(__CUDACC__)
// Records are read through L2 (the plan kernel that wrote them may have run
// concurrently with this grid's launch).
template <typename T>
__device__ __forceinline__ T load_record(const T *base, int rec) {
    static_assert(sizeof(T) % 16 == 0, "record size");
    T r;
    const int4 *src = reinterpret_cast<const int4 *>(base + rec);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(T) / 16); ++i)
        reinterpret_cast<int4 *>(&r)[i] = __ldcg(src + i);
    return r;
}
template <typename T>
__device__ __forceinline__ void store_record(T *base, int rec, const T &r) {
    int4 *dst = reinterpret_cast<int4 *>(base + rec);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(T) / 16); ++i)
        dst[i] = reinterpret_cast<const int4 *>(&r)[i];
}
#endif

// Byte offsets of the workspace regions (same computation on host and device).
struct WsLayout {
    size_t header, counters, short_items, long_items, partial_o, partial_lse, extra_o, extra_lse;
    size_t prefix_o, prefix_lse;    // cascade prefix pass: split states [rows][D], [rows]
    size_t stage_base, stage_list;  // fp8 staging bookkeeping ([num_seqs] each)
    size_t total;
    int max_short, max_long, cap_rows, num_counters;
};

// Kernel parameter blocks -----------------------------------------------------
struct ShortParams {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    float *lse;
    const int *block_tables;
    int bt_stride;
    const int *qsl, *ctx, *seq_lens;
    int num_q_heads, num_kv_heads, group, block_size, num_blocks, kv_rows;
    float scale_log2;
    PlanHeader *hdr;
    const ShortItem *items;
    int *counters;
    float *partial_o, *partial_lse;
    // if set, every row's final state is written as fp32 (o normalised
    // [row][D], lse [row] into `lse`) instead of bf16 out: cascade decode's
    // suffix state, merged with the prefix state by the fold kernel
    float *out_f32;
    const float *k_scale, *v_scale;    // fp8 pool: per-kv-head dequantisation scales
    int no_start_wait;  // launched after the step's first tensor-core grid (see LongParams)
    unsigned *status;
    int num_seqs, num_q_tokens;  // sizes of the metadata arrays and of q (L2 warm-up)
    int max_items;               // work-record capacity of the workspace (>= 1)
    int claim_ahead;  // ring stages before an item's end at which the next is claimed (0: at its start)
    int test_stall;   // test hook: CTA 0's producer stops after its first stage
};

struct LongParams {
    __nv_bfloat16 *out;
    float *lse;
    float *out_f32;          // if set, final output is written as fp32 state here
    const int *block_tables;  // per-request tables, or the prefix block list
    int bt_stride;            // 0 in prefix mode
    const int *qsl, *ctx, *seq_lens;
    int num_q_tokens, num_q_heads, num_kv_heads, group, q_tile_tokens, block_size, num_blocks,
        kv_rows;
    float scale_log2;
    int prefix_mode;  // 1: non-causal shared prefix, items implicit
    int prefix_len, prefix_nsplit, prefix_split_keys, prefix_q_tiles;
    int states_only;  // 1: every item writes its split state, even when unsplit
    PlanHeader *hdr;
    const LongItem *items;
    float *partial_o, *partial_lse;
    unsigned *status;
    // fp8 pool with a bf16 staging copy: request b's key block j is staging
    // block stage_base[b] + j (decoded codes, unscaled); scores are scaled by
    // k_scale[h] and outputs by v_scale[h].  NULL for a bf16 pool.
    const int *stage_base;
    const float *k_scale, *v_scale;
    // Step mode launch protocol.  dynamic: items from the step's counter
    // (hdr->long_next) through a per-CTA queue, so several launches can share
    // the work; wait_start: wait for the previous grid (the plan) before
    // reading anything; first_done: completion counter of the step's first
    // tensor-core launch -- that launch (first_ctas < 0) counts its CTAs,
    // the last launch (first_ctas = the first launch's grid) completes only
    // after all of them.
    int dynamic, wait_start;
    int *first_done;
    int first_ctas;
    unsigned long long *tile_counter;  // if set: += 128-key tiles whose Q K^T was issued
    // 1: launched as a programmatic dependent of the split-KV kernel of the
    // same step.  The kernel then reads nothing but the plan's output (and
    // the step's inputs) before its last instruction, where it waits for the
    // split-KV grid so that its own completion still orders the stream.
    int overlap_prev;
};

struct PlanParams {
    const int *qsl, *ctx, *seq_lens;
    int num_seqs, num_q_tokens, num_kv_heads, group, q_tile_tokens;
    int short_max_rows;  // q_len*group <= this -> split-KV kernel
    int piece_tokens;    // a split-KV request is cut into pieces of this many tokens
    // fp8 pool: long requests (q_len * group > kShortMaxRows) get a bf16
    // staging copy of their blocks, in request order while stage_cap blocks
    // last; stage_base[b] = first staging block or -1, stage_list = staged
    // requests in order.  stage_cap = 0: no staging (all rows split-KV).
    int fp8, stage_cap, block_size;
    int *stage_base, *stage_list;
    int split_stages;    // 0 = automatic
    int target_items;    // automatic split aims at about this many split-KV items
    int num_ctas;        // persistent split-KV CTAs of the launch
    PlanHeader *hdr;
    ShortItem *short_items;
    LongItem *long_items;
    int *counters;
    int max_short, max_long, cap_rows, num_counters;
    unsigned *status;
};

// Merge of the prefix pass's split states: item (kv head h, query tile qt,
// split s) wrote row r of its tile at partial row
// ((h * q_tiles + qt) * nsplit + s) * 128 + r.
struct PrefixFoldParams {
    const float *partial_o, *partial_lse;
    // optional further state per row ([T*Hq][D] fp32 normalised, [T*Hq] lse):
    // cascade decode's suffix state
    const float *extra_o, *extra_lse;
    int nsplit, q_tiles, pairs, group, q_tile_tokens, num_q_tokens, num_q_heads;
    __nv_bfloat16 *out;  // bf16 result, or
    float *out_f32;      // fp32 result (a state for the suffix pass)
    float *lse;          // may be NULL
};

// Launch configuration with the programmatic-stream-serialisation attribute
// (programmatic dependent launch): the kernel may be scheduled while the
// previous kernel of the stream is still running, and must call pdl_wait()
// before it touches anything that kernel (or an earlier one) produces.
struct PdlLaunch {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl = true) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
    }
    PdlLaunch(const PdlLaunch &) = delete;
    PdlLaunch &operator=(const PdlLaunch &) = delete;
};

// Runs fn() (a cudaError_t-returning set-up step such as a function
// attribute) once per device: attributes set with cudaFuncSetAttribute belong
// to the function's instance on the device current at the call, so a second
// GPU in the same process needs its own.
struct PerDeviceOnce {
    std::mutex mu;
    uint64_t mask = 0;  // bit d: done on device d (devices 0..63)
};
template <typename F>
int once_per_device(PerDeviceOnce &once, F &&fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(once.mu);
    if ((once.mask >> dev) & 1u) return PA_OK;
    if (fn() != cudaSuccess) return PA_ERR_CUDA;
    once.mask |= 1ull << dev;
    return PA_OK;
}

// Every kernel launch of the library goes through launch_kernel, which keeps
// the process-wide count that pa_kernel_launches() reports.
void count_launch();
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const PdlLaunch &l, void (*kernel)(KArgs...), Args &&...args) {
    const cudaError_t e = cudaLaunchKernelEx(&l.cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) count_launch();
    return e;
}

// Host-side launchers (each defined next to its kernel).
int launch_write_kv(const void *k, const void *v, const int64_t *slots, int num_tokens,
                    const pa_kv_desc *kv, unsigned *status, cudaStream_t s);
// Decodes the e4m3 blocks of the staged requests (plan output) into the
// bf16 staging pool; grid-stride over staging blocks.
int launch_stage_fp8(const pa_kv_desc *kv, const int32_t *block_tables, int32_t bt_stride,
                     const PlanHeader *hdr, const int *stage_base, const int *stage_list,
                     void *stage_k, void *stage_v, unsigned *status, int grid, cudaStream_t s);
// The shared prefix's n e4m3 blocks decoded to bf16 staging blocks 0..n-1
// (cascade decode on an e4m3 pool); ident[k] = k is the staged block list.
int launch_stage_prefix_fp8(const pa_kv_desc *kv, const int32_t *prefix_blocks, int n,
                            int32_t *ident, void *stage_k, void *stage_v, unsigned *status,
                            int grid, cudaStream_t s);
int launch_plan(const PlanParams &p, cudaStream_t s);
int launch_short(const ShortParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                 int head_dim, bool fp8, int grid, cudaStream_t s);
int short_max_ctas_per_sm(int head_dim, bool fp8);
int launch_long(const LongParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                const CUtensorMap &tv, int head_dim, int grid, cudaStream_t s);
int launch_prefix_fold(const PrefixFoldParams &f, int head_dim, cudaStream_t s);
int launch_merge(const void *oa, const float *la, const void *ob, const float *lb, int n,
                 int heads, int head_dim, void *out, float *lse_out, cudaStream_t s);
size_t short_smem_bytes(int head_dim);
// One attention step whose scratch is a caller-provided region of fixed size
// (defined in pa_api.cu, used by pa_static.cu).
int attention_in_fixed_workspace(const void *q, const pa_kv_desc *kv,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *query_start_loc, const int32_t *context_lens,
                                 const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_tokens,
                                 int32_t num_q_heads, float scale, void *out, float *lse,
                                 void *scratch, size_t scratch_bytes, cudaStream_t s);
// Record `msg` as the calling thread's last error message; returns `code`.
int set_error_message(int code, const char *msg);
size_t long_smem_bytes(int head_dim);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Atomic add at GPU scope with acquire-release semantics.  It publishes the
// writes ordered before it (the CTA's, through a preceding CTA barrier) and,
// to the thread that reads the final count, makes visible what the other
// adders published.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *ptr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(ptr), "r"(v)
                 : "memory");
    return old;
}

__device__ __forceinline__ void flag_status(unsigned *status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

// 2^x by the hardware approximation (one instruction; relative error of a
// few units in the last place of fp32, subnormal results flushed to zero):
// the softmax exponentials, whose results feed bf16 / f16 MMA operands.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
// Programmatic dependent launch: wait until the previous grid of the stream
// has completed and its memory is visible (a no-op for a plain launch), and
// allow the next grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up (returning false and raising *abort) when the
// barrier phase has not completed within kWaitTimeoutNs, or as soon as
// another thread of the CTA has raised *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            *abort = 1;
            return false;
        }
    }
}
// Warp-wide bounded wait: lane 0 polls (bounded, see mbar_wait), then every
// lane tests the now-complete phase itself so that each thread has its own
// acquire of the barrier, and __syncwarp keeps the compiler from moving any
// lane's later loads or stores above the wait.  Returns the same value in
// all lanes.
__device__ __forceinline__ bool warp_mbar_wait(uint64_t *bar, uint32_t parity,
                                               volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    __syncwarp();
    return ok != 0;
}
// Non-blocking test of a barrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait that polls without suspending the thread, for waits whose
// wake-up latency sits on a warp's critical path and whose warps have few
// neighbours competing for issue slots (the split-KV kernel's producer and
// consumers: measured 0.4 us median between a slot's release and the
// suspended producer noticing it).  Same bound and abort protocol.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity,
                                               volatile int *abort) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_test_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            *abort = 1;
            return false;
        }
    }
}
// warp_mbar_wait with the polling wait above.
__device__ __forceinline__ bool warp_mbar_wait_spin(uint64_t *bar, uint32_t parity,
                                                    volatile int *abort) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_spin(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    __syncwarp();
    return ok != 0;
}
// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > 100000000ull) break;
    }
}

// TMA --------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *tm, int c0, int c1,
                                            int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
// L2 prefetch of slice `part` of `parts` of [base, base + bytes) by the 32
// lanes of a warp, in bulk pieces of at most 4 KB.  Only whole 16-byte units
// inside the range are named (the bulk prefetch needs 16-byte alignment).
// A prefetch is a hint: it moves nothing into registers or shared memory.
__device__ __forceinline__ void l2_prefetch_slice(const void *base, size_t bytes, int part,
                                                  int parts, int lane) {
    const uint64_t lo = (reinterpret_cast<uint64_t>(base) + 15) & ~15ull;
    const uint64_t hi = (reinterpret_cast<uint64_t>(base) + bytes) & ~15ull;
    if (!base || hi <= lo || parts <= 0) return;
    const uint64_t per = (((hi - lo) + parts - 1) / parts + 15) & ~15ull;
    const uint64_t s = lo + per * static_cast<uint64_t>(part);
    if (s >= hi) return;
    const uint64_t e = s + per < hi ? s + per : hi;
    for (uint64_t a = s + static_cast<uint64_t>(lane) * 4096; a < e; a += 32 * 4096) {
        const uint32_t n = static_cast<uint32_t>(e - a < 4096 ? e - a : 4096);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(n) : "memory");
    }
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier among `count` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Offset of 16-byte column `chunk` (0..7) of row `row` inside a tile written
// by TMA with 128-byte swizzling (rows of 128 bytes, 1024-byte aligned base):
// the hardware XORs the chunk index with the row index modulo 8.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Warp-level tensor core (memory-bound split-KV kernel) ---------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// f16 forms for the fp8 KV pool: K/V codes decode exactly to f16.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// lo -> bits 0..15, hi -> bits 16..31
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// two bf16 (lo, hi halves of v) -> two f16, same positions
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}
// four e4m3 codes (bytes 0..3 of w) -> two f16x2: lo = (byte 0, byte 1),
// hi = (byte 2, byte 3), each first code in the low half; exact, since every
// e4m3 value is an f16 value
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}
// transpose of an 8x8 b16 matrix held as one mma fragment register per lane
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
__device__ __forceinline__ uint32_t byte_perm(uint32_t x, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(x), "r"(sel));
    return r;
}

// tcgen05 / TMEM -------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor (tcgen05): start address, leading- and
// stride-dimension byte offsets (all >> 4), descriptor version 1 at bit 46,
// swizzle mode in bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}
// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulate.
// b_mn_major: B operand stored N-contiguous (e.g. V rows for P*V).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
    return (1u << 4)                                  // D format: f32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | (static_cast<uint32_t>(b_mn_major) << 16)  // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same MMA with the A operand (M x K, one row per TMEM lane, two 16-bit
// elements per 32-bit column) read from tensor memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 lanes x 32 columns of 32-bit TMEM cells: thread i gets lane (base+i),
// columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
// One 32-bit TMEM cell per thread (lane = thread, one column).
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t (&r)[1]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r[0]) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, const uint32_t (&r)[1]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r[0])
                 : "memory");
}

#endif  // __CUDACC__

}  // namespace pa
