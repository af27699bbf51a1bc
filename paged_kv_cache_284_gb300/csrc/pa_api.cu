// pa_api.cu -- the C ABI of libpa (declared in include/pa.h): argument checks,
// TMA tensor maps, workspace layout and the launch sequence of one step.
// Every step of the path runs in this library's kernels; nothing here
// computes on the host beyond integer bookkeeping.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "pa_internal.cuh"

using namespace pa;

// Per-device status word (PA_DEV_* bits).  Host code passes its device
// address to the kernels; pa_read_device_status reads it back.
__device__ unsigned int g_pa_status;

namespace {

thread_local char g_err[256] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int short_ctas_per_sm[3] = {0, 0, 0};  // bf16 head_dim 64, bf16 128, fp8 128
    unsigned *status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(PA_ERR_CUDA, "no current CUDA device");
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        void *sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_pa_status) != cudaSuccess)
            return fail(PA_ERR_CUDA, "cudaGetSymbolAddress(status) failed");
        d.status = static_cast<unsigned *>(sym);
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(PA_ERR_CUDA, "cannot query SM count");
        d.short_ctas_per_sm[0] = short_max_ctas_per_sm(64, false);
        d.short_ctas_per_sm[1] = short_max_ctas_per_sm(128, false);
        d.short_ctas_per_sm[2] = short_max_ctas_per_sm(128, true);
        d.ready = true;
    }
    *out = &d;
    return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of one cache array: rows = (block, kv head, offset) flattened,
// head_dim columns; boxes of 16 rows x 128 bytes (64 bf16 or 128 e4m3
// columns), 128-byte swizzle.
int make_kv_map(CUtensorMap *m, void *base, int64_t rows, int head_dim, bool fp8) {
    auto fn = encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const int esize = fp8 ? 1 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * esize};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(kChunkKeys)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : fail(PA_ERR_CUDA, "KV tensor map encode failed (%d)", (int)r);
}

// 3-D view of q [tokens][q heads][head_dim]; a box is 64 dims x group heads x
// tile tokens, i.e. the 128 (token, head) rows of one tensor-core tile.
int make_q_map(CUtensorMap *m, const void *q, int tokens, int heads, int head_dim, int group,
               int tile_tokens) {
    auto fn = encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(tokens > 0 ? tokens : 1)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                             static_cast<cuuint64_t>(heads) * head_dim * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tile_tokens)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : fail(PA_ERR_CUDA, "Q tensor map encode failed (%d)", (int)r);
}

std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_test_stall{PA_TEST_STALL_NONE};  // pa_set_test_stall
std::atomic<uint64_t *> g_tile_counter{nullptr};     // pa_set_tile_counter

// Profiling hook state (pa_set_profile_events).
void *g_prof[4][2] = {};
std::mutex g_prof_mu;

struct ProfScope {
    int which;
    cudaStream_t s;
    void *end;
    ProfScope(int w, cudaStream_t st) : which(w), s(st), end(nullptr) {
        void *start;
        {
            std::lock_guard<std::mutex> lock(g_prof_mu);
            start = g_prof[w][0];
            end = g_prof[w][1];
        }
        if (start) cudaEventRecord(static_cast<cudaEvent_t>(start), s);
    }
    ~ProfScope() {
        if (end) cudaEventRecord(static_cast<cudaEvent_t>(end), s);
    }
};

// True while per-kernel profiling events are set: the step then launches its
// kernels one after the other so that each event pair times one kernel.
// Fewest query tokens for which a step runs its split-KV and tensor-core
// kernels side by side (below it they run one after the other).
constexpr int kSideBySideMinTokens = 512;

bool profiling_active() {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    return g_prof[PA_KERNEL_SPLIT_KV][0] || g_prof[PA_KERNEL_TENSOR_CORE][0];
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int q_tile_tokens(int group) { return group <= kLongRows ? kLongRows / group : 0; }

// Query tokens per split-KV piece (a piece fills at most kShortMaxRows rows),
// and a bound on the pieces of a step with these sizes.
int piece_tokens_for(int group) { return std::max(1, kShortMaxRows / std::max(1, group)); }
int pieces_bound(int num_seqs, int num_q_tokens, int group) {
    const int pt = piece_tokens_for(group);
    return num_seqs + (num_q_tokens + pt - 1) / pt;
}

// prefix_rows > 0: room for the cascade prefix pass's split states;
// with_extra: room for cascade decode's fp32 suffix state ([T*Hq] rows).
WsLayout make_layout(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads,
                     int head_dim, int prefix_rows, bool with_extra) {
    WsLayout L{};
    const int group = num_q_heads / num_kv_heads;
    const int tq = q_tile_tokens(group);
    const int pieces = pieces_bound(num_seqs, num_q_tokens, group);
    L.max_short = num_kv_heads * (num_seqs * 8 + pieces) + 4096;
    L.max_long = num_kv_heads * ((num_q_tokens + tq - 1) / tq + num_seqs);
    L.cap_rows = L.max_short * 4;
    L.num_counters = num_kv_heads * std::max(1, pieces);
    size_t off = 0;
    L.header = off;
    off = align256(off + sizeof(PlanHeader));
    L.counters = off;
    off = align256(off + sizeof(int) * static_cast<size_t>(L.num_counters));
    L.short_items = off;
    off = align256(off + sizeof(ShortItem) * static_cast<size_t>(L.max_short));
    L.long_items = off;
    off = align256(off + sizeof(LongItem) * static_cast<size_t>(L.max_long));
    L.partial_o = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(L.cap_rows) * head_dim);
    L.partial_lse = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(L.cap_rows));
    L.stage_base = off;
    off = align256(off + sizeof(int) * static_cast<size_t>(num_seqs > 0 ? num_seqs : 1));
    L.stage_list = off;
    off = align256(off + sizeof(int) * static_cast<size_t>(num_seqs > 0 ? num_seqs : 1));
    if (with_extra) {
        const size_t rows = static_cast<size_t>(num_q_tokens) * num_q_heads;
        L.extra_o = off;
        off = align256(off + sizeof(float) * rows * head_dim);
        L.extra_lse = off;
        off = align256(off + sizeof(float) * rows);
    }
    if (prefix_rows > 0) {
        L.prefix_o = off;
        off = align256(off + sizeof(float) * static_cast<size_t>(prefix_rows) * head_dim);
        L.prefix_lse = off;
        off = align256(off + sizeof(float) * static_cast<size_t>(prefix_rows));
    }
    L.total = off;
    return L;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_kv(const pa_kv_desc *kv) {
    if (!kv) return fail(PA_ERR_INVALID_ARG, "kv descriptor is NULL");
    if (!kv->k_cache || !kv->v_cache) return fail(PA_ERR_INVALID_ARG, "cache pointer is NULL");
    if (!aligned(kv->k_cache, 16) || !aligned(kv->v_cache, 16))
        return fail(PA_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
    if (kv->num_blocks <= 0 || kv->num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "num_blocks and num_kv_heads must be positive");
    if (kv->head_dim != 64 && kv->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not built (64 or 128)", kv->head_dim);
    if (kv->block_size <= 0 || kv->block_size % 16 != 0 || kv->block_size > 256)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d: need a multiple of 16, at most 256",
                    kv->block_size);
    if (kv->reserved != 0) return fail(PA_ERR_INVALID_ARG, "pa_kv_desc.reserved must be 0");
    if (kv->kv_dtype == PA_KV_FP8_E4M3) {
        if (kv->head_dim != 128)
            return fail(PA_ERR_UNSUPPORTED, "fp8 KV pool: head_dim %d not built (128)", kv->head_dim);
        if (!kv->k_scale || !kv->v_scale || !aligned(kv->k_scale, 4) || !aligned(kv->v_scale, 4))
            return fail(PA_ERR_INVALID_ARG, "fp8 KV pool needs 4-byte aligned k_scale and v_scale");
    } else if (kv->kv_dtype != PA_KV_BF16) {
        return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d unknown", kv->kv_dtype);
    }
    const int64_t rows = static_cast<int64_t>(kv->num_blocks) * kv->num_kv_heads * kv->block_size;
    if (rows >= (static_cast<int64_t>(1) << 31) - 256)
        return fail(PA_ERR_UNSUPPORTED, "pool too large: %lld cache rows", (long long)rows);
    return PA_OK;
}

int check_heads(const pa_kv_desc *kv, int num_q_heads) {
    if (num_q_heads <= 0 || num_q_heads % kv->num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    num_q_heads, kv->num_kv_heads);
    const int group = num_q_heads / kv->num_kv_heads;
    if (group > kLongRows || group > 255)
        return fail(PA_ERR_UNSUPPORTED, "group size %d too large", group);
    return PA_OK;
}

int64_t kv_rows(const pa_kv_desc *kv) {
    return static_cast<int64_t>(kv->num_blocks) * kv->num_kv_heads * kv->block_size;
}

struct StepMaps {
    CUtensorMap q, k, v;
};

// bf16 staging copy of the long requests' blocks of an fp8 pool: the part of
// the caller's workspace beyond the step's own layout (cap blocks for K and
// for V, [cap][Hkv][bs][d] each).
struct Staging {
    int cap = 0;
    void *k = nullptr, *v = nullptr;
    CUtensorMap tk, tv;
};

size_t stage_block_bytes(const pa_kv_desc *kv) {
    return static_cast<size_t>(kv->num_kv_heads) * kv->block_size * kv->head_dim * 2;
}

// Carves the staging area out of workspace bytes [used, total).
int make_staging(Staging *st, const pa_kv_desc *kv, uint8_t *ws, size_t used, size_t total) {
    st->cap = 0;
    if (kv->kv_dtype != PA_KV_FP8_E4M3 || !ws) return PA_OK;
    const size_t start = align256(used);
    const size_t blk = stage_block_bytes(kv);
    if (total < start + 512 + 2 * blk) return PA_OK;
    size_t cap = (total - start - 512) / (2 * blk);
    const size_t max_rows = (static_cast<size_t>(1) << 31) - 256;
    cap = std::min(cap, max_rows / (static_cast<size_t>(kv->num_kv_heads) * kv->block_size));
    cap = std::min<size_t>(cap, 1u << 28);
    st->cap = static_cast<int>(cap);
    st->k = ws + start;
    st->v = ws + start + align256(cap * blk);
    const int64_t rows = static_cast<int64_t>(cap) * kv->num_kv_heads * kv->block_size;
    int rc = make_kv_map(&st->tk, st->k, rows, kv->head_dim, false);
    if (rc == PA_OK) rc = make_kv_map(&st->tv, st->v, rows, kv->head_dim, false);
    return rc;
}

// Cascade decode on an e4m3 pool: the shared prefix decoded to bf16 for the
// tensor-core prefix pass, in the workspace beyond the call's own layout:
// the identity block list ident[k] = k (n int32), then n staging blocks of K
// and of V.  n = 0: a bf16 pool or an empty prefix (nothing staged).
struct PrefixStage {
    int n = 0;
    int32_t *ident = nullptr;
    Staging stg;
};

size_t prefix_stage_bytes(int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t prefix_len) {
    const int64_t n = (static_cast<int64_t>(prefix_len) + block_size - 1) / block_size;
    if (n == 0) return 0;
    const size_t blk = static_cast<size_t>(num_kv_heads) * block_size * head_dim * 2;
    return align256(sizeof(int32_t) * static_cast<size_t>(n)) +
           2 * align256(static_cast<size_t>(n) * blk) + 768;
}

int make_prefix_stage(PrefixStage *ps, const pa_kv_desc *kv, int32_t prefix_len, uint8_t *ws,
                      size_t used, size_t total) {
    ps->n = 0;
    if (kv->kv_dtype != PA_KV_FP8_E4M3 || prefix_len == 0) return PA_OK;
    const int n = static_cast<int>((static_cast<int64_t>(prefix_len) + kv->block_size - 1) /
                                   kv->block_size);
    const size_t start = align256(used);
    const size_t need =
        start + prefix_stage_bytes(kv->num_kv_heads, kv->head_dim, kv->block_size, prefix_len);
    if (total < need)
        return fail(PA_ERR_WORKSPACE,
                    "an e4m3 pool's shared prefix is decoded to bf16 in the workspace: it needs "
                    "%zu bytes (pa_cascade_workspace_size + pa_cascade_fp8_staging_bytes), got %zu",
                    need, total);
    ps->ident = reinterpret_cast<int32_t *>(ws + start);
    int rc = make_staging(&ps->stg, kv, ws, start + align256(sizeof(int32_t) * n), total);
    if (rc != PA_OK) return fail(rc, "prefix staging map failed");
    if (ps->stg.cap < n) return fail(PA_ERR_WORKSPACE, "prefix staging area too small");
    ps->n = n;
    return PA_OK;
}

// Decodes the prefix into the staging area (a launch on `s`) and points the
// prefix pass at it: the identity list, the staging blocks and the pool's
// scales.  The pass's K and V tensor maps become *tk and *tv.
int stage_prefix(const PrefixStage &ps, const pa_kv_desc *kv, const int32_t *prefix_blocks,
                 LongParams *lp, const CUtensorMap **tk, const CUtensorMap **tv,
                 DeviceInfo *dev, cudaStream_t s) {
    if (ps.n == 0) return PA_OK;
    const int rc = launch_stage_prefix_fp8(kv, prefix_blocks, ps.n, ps.ident, ps.stg.k,
                                           ps.stg.v, dev->status, 2 * dev->sms, s);
    if (rc != PA_OK) return fail(rc, "prefix staging launch failed");
    lp->block_tables = ps.ident;
    lp->num_blocks = ps.stg.cap;
    lp->kv_rows = ps.stg.cap * kv->num_kv_heads * kv->block_size;
    lp->k_scale = kv->k_scale;
    lp->v_scale = kv->v_scale;
    *tk = &ps.stg.tk;
    *tv = &ps.stg.tv;
    return PA_OK;
}

int make_maps(StepMaps *m, const void *q, const pa_kv_desc *kv, int tokens, int heads) {
    const int group = heads / kv->num_kv_heads;
    const bool fp8 = kv->kv_dtype == PA_KV_FP8_E4M3;
    int rc = make_kv_map(&m->k, kv->k_cache, kv_rows(kv), kv->head_dim, fp8);
    if (rc == PA_OK) rc = make_kv_map(&m->v, kv->v_cache, kv_rows(kv), kv->head_dim, fp8);
    if (rc == PA_OK)
        rc = make_q_map(&m->q, q, tokens, heads, kv->head_dim, group, q_tile_tokens(group));
    return rc;
}

int prefix_plan(int T, int prefix_len, int num_kv_heads, int group, int sms, int *q_tiles,
                int *nsplit, int *split_keys) {
    const int tq = q_tile_tokens(group);
    *q_tiles = (T + tq - 1) / tq;
    const int tiles = (prefix_len + kLongKeys - 1) / kLongKeys;
    const int pairs = num_kv_heads * *q_tiles;
    // the prefix kernel is persistent (one CTA per SM): split the key range so
    // that every (kv head, query tile, split) item gets an SM of its own
    int ns = std::max(1, sms / std::max(1, pairs));
    ns = std::max(1, std::min(ns, std::min(64, tiles)));
    const int per = std::max(1, (tiles + ns - 1) / ns);  // KV tiles per split (an empty prefix: 1)
    *split_keys = per * kLongKeys;
    *nsplit = (prefix_len + *split_keys - 1) / *split_keys;
    if (*nsplit < 1) *nsplit = 1;
    return PA_OK;
}

// Parameters of the shared-prefix ("multi-query") pass: items are (kv head,
// query tile, key split), implicit in the index; split states go to
// (split_o, split_lse) at row (pair * nsplit + split) * 128 + r.
LongParams prefix_params(const pa_kv_desc *kv, const int32_t *prefix_blocks, int32_t prefix_len,
                         int32_t T, int32_t Hq, float scale, int q_tiles, int nsplit,
                         int split_keys, float *split_o, float *split_lse, DeviceInfo *dev) {
    const int group = Hq / kv->num_kv_heads;
    LongParams lp{};
    lp.block_tables = prefix_blocks;
    lp.bt_stride = 0;
    lp.num_q_tokens = T;
    lp.num_q_heads = Hq;
    lp.num_kv_heads = kv->num_kv_heads;
    lp.group = group;
    lp.q_tile_tokens = q_tile_tokens(group);
    lp.block_size = kv->block_size;
    lp.num_blocks = kv->num_blocks;
    lp.kv_rows = static_cast<int>(kv_rows(kv));
    lp.scale_log2 = scale * 1.4426950408889634f;
    lp.prefix_mode = 1;
    lp.prefix_len = prefix_len;
    lp.prefix_nsplit = nsplit;
    lp.prefix_split_keys = split_keys;
    lp.prefix_q_tiles = q_tiles;
    lp.partial_o = split_o;
    lp.partial_lse = split_lse;
    lp.status = dev->status;
    return lp;
}

// Cascade decode: the shared prefix and where its states and the suffix
// states live in the workspace.
struct CascadeArgs {
    const int32_t *prefix_blocks;
    int32_t prefix_len;
    const PrefixStage *ps;  // an e4m3 pool's prefix, decoded to bf16 (ps->n = 0: none)
    float *prefix_o, *prefix_lse;  // prefix split states
    float *suffix_o, *suffix_lse;  // suffix state per row, fp32
};

// The step's new K/V rows, for the call that writes them and attends.
struct NewRows {
    const void *k, *v;
    const int64_t *slots;
    int32_t num_tokens;
};

// Checks of pa_write_kv's arguments; num_tokens == 0 needs no pointers.
int check_new_rows(const NewRows &nr) {
    if (nr.num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (nr.num_tokens == 0) return PA_OK;
    if (!nr.k || !nr.v || !nr.slots) return fail(PA_ERR_INVALID_ARG, "NULL input");
    if (!aligned(nr.k, 16) || !aligned(nr.v, 16))
        return fail(PA_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    return PA_OK;
}

// Runs the planner, the split-KV kernel and the tensor-core kernel of one
// step on `s`.  With `casc` (cascade decode, all rows short) the step is
// the unique-suffix pass, run side by side with the shared-prefix pass.
// With `fresh`, the step's new rows are written into the cache first.
int run_step(const void *q, const pa_kv_desc *kv, const int32_t *block_tables, int32_t max_blocks,
             const int32_t *qsl, const int32_t *ctx, const int32_t *seq_lens, int32_t num_seqs,
             int32_t T, int32_t Hq, float scale, void *out, float *lse, uint8_t *ws,
             const WsLayout &L, int short_max_rows, int split_keys, const CascadeArgs *casc,
             bool forbid_long, const StepMaps &maps, const Staging &stg, DeviceInfo *dev,
             cudaStream_t s, const NewRows *fresh = nullptr) {
    const int D = kv->head_dim;
    const int group = Hq / kv->num_kv_heads;
    const int tq = q_tile_tokens(group);
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(ws + L.header);

    PlanParams pp{};
    pp.qsl = qsl;
    pp.ctx = ctx;
    pp.seq_lens = seq_lens;
    pp.num_seqs = num_seqs;
    pp.num_q_tokens = T;
    pp.num_kv_heads = kv->num_kv_heads;
    pp.group = group;
    pp.q_tile_tokens = tq;
    // An fp8 pool runs short rows on the split-KV kernel; long requests run on
    // the tensor-core kernel over a bf16 staging copy while staging blocks
    // last, and as split-KV pieces of piece_tokens query tokens otherwise
    // (all of them when the workspace has no staging area).
    const bool fp8 = kv->kv_dtype == PA_KV_FP8_E4M3;
    const bool staged = fp8 && stg.cap > 0;
    if (fp8 && !staged) forbid_long = true;
    pp.short_max_rows = forbid_long ? 0x7fffffff : short_max_rows;
    pp.piece_tokens = std::max(1, std::min(pp.short_max_rows, kShortMaxRows) / group);
    pp.fp8 = fp8 ? 1 : 0;
    pp.stage_cap = staged ? stg.cap : 0;
    pp.block_size = kv->block_size;
    pp.stage_base = staged ? reinterpret_cast<int *>(ws + L.stage_base) : nullptr;
    pp.stage_list = staged ? reinterpret_cast<int *>(ws + L.stage_list) : nullptr;
    pp.split_stages = split_keys / kStageKeys;
    const int short_grid = dev->sms * dev->short_ctas_per_sm[fp8 ? 2 : (D == 128 ? 1 : 0)];
    pp.target_items = kSplitItemsPerCta * short_grid;
    pp.num_ctas = short_grid;
    pp.hdr = hdr;
    pp.short_items = reinterpret_cast<ShortItem *>(ws + L.short_items);
    pp.long_items = reinterpret_cast<LongItem *>(ws + L.long_items);
    pp.counters = reinterpret_cast<int *>(ws + L.counters);
    pp.max_short = L.max_short;
    pp.max_long = L.max_long;
    pp.cap_rows = L.cap_rows;
    pp.num_counters = L.num_counters;
    pp.status = dev->status;
    int rc;
    if (fresh && fresh->num_tokens > 0) {
        // The step's new rows first, as pa_write_kv does: its kernel runs as a
        // programmatic dependent ahead of the planner and is off the step's
        // critical path.  (Writing them from copy blocks in the planner's
        // grid measured no faster on an 8-request decode step and slower on
        // large ones.)
        ProfScope prof(PA_KERNEL_WRITE_KV, s);
        rc = launch_write_kv(fresh->k, fresh->v, fresh->slots, fresh->num_tokens, kv, dev->status,
                             s);
        if (rc != PA_OK) return fail(rc, "write_kv launch failed");
    }
    {
        ProfScope prof(PA_KERNEL_PLAN, s);
        rc = launch_plan(pp, s);
    }
    if (rc != PA_OK) return fail(rc, "plan launch failed");
    if (staged) {
        rc = launch_stage_fp8(kv, block_tables, max_blocks, hdr, pp.stage_base, pp.stage_list,
                              stg.k, stg.v, dev->status, 2 * dev->sms, s);
        if (rc != PA_OK) return fail(rc, "fp8 staging copy launch failed");
    }

    ShortParams sp{};
    sp.q = static_cast<const __nv_bfloat16 *>(q);
    sp.out = static_cast<__nv_bfloat16 *>(out);
    sp.lse = lse;
    sp.block_tables = block_tables;
    sp.bt_stride = max_blocks;
    sp.qsl = qsl;
    sp.ctx = ctx;
    sp.seq_lens = seq_lens;
    sp.num_q_heads = Hq;
    sp.num_kv_heads = kv->num_kv_heads;
    sp.group = group;
    sp.block_size = kv->block_size;
    sp.num_blocks = kv->num_blocks;
    sp.kv_rows = static_cast<int>(kv_rows(kv));
    sp.scale_log2 = scale * 1.4426950408889634f;
    sp.hdr = hdr;
    sp.items = pp.short_items;
    sp.counters = pp.counters;
    sp.partial_o = reinterpret_cast<float *>(ws + L.partial_o);
    sp.partial_lse = reinterpret_cast<float *>(ws + L.partial_lse);
    sp.out_f32 = nullptr;
    sp.k_scale = fp8 ? kv->k_scale : nullptr;
    sp.v_scale = fp8 ? kv->v_scale : nullptr;
    sp.status = dev->status;
    sp.num_seqs = num_seqs;
    sp.num_q_tokens = T;
    sp.max_items = L.max_short;
    sp.claim_ahead = kClaimAheadStages;
    const int stall = g_test_stall.load(std::memory_order_relaxed);
    sp.test_stall = stall == PA_TEST_STALL_SPLIT_KV ? 1 : 0;

    if (casc) {
        // Cascade decode ([AI] §02.1): the shared-prefix pass (tensor cores,
        // compute-heavy, each prefix tile read once per 128 query rows) and
        // the unique-suffix pass (split-KV, HBM-bound) have disjoint inputs,
        // so they run side by side like the two halves of a mixed step: a
        // first prefix grid waits for the plan and lets the split-KV grid in
        // on the other SMs; a second prefix grid takes SMs over as split-KV
        // CTAs finish (both pull prefix items from the step's counter) and
        // completes after both.  The split-KV grid writes
        // each row's suffix state in fp32; the fold kernel merges it with the
        // prefix split states into out and lse.
        // The prefix pass's items are cut for one round on about 36 % of the
        // SMs (the first grid takes them all); the split-KV grid streams the
        // suffixes on the rest.  Measured on 64 requests x an 8192-token
        // prefix, us per call by share: 28 % 73.9 (too few splits), 32 %
        // 63.4, 36 % 63.1-63.5, 42 % 64.6, 48 % 64.5, 54 % 67.4.
        int q_tiles, nsplit, split_keys_p;
        const int prefix_sms = std::max(1, (dev->sms * 36 + 50) / 100);
        prefix_plan(T, casc->prefix_len, kv->num_kv_heads, group, prefix_sms, &q_tiles, &nsplit,
                    &split_keys_p);
        LongParams cp = prefix_params(kv, casc->prefix_blocks, casc->prefix_len, T, Hq, scale,
                                      q_tiles, nsplit, split_keys_p, casc->prefix_o,
                                      casc->prefix_lse, dev);
        // an e4m3 pool: the prefix decoded to bf16 first (after the plan; the
        // first prefix grid waits for it)
        const CUtensorMap *ptk = &maps.k, *ptv = &maps.v;
        rc = stage_prefix(*casc->ps, kv, casc->prefix_blocks, &cp, &ptk, &ptv, dev, s);
        if (rc != PA_OK) return rc;
        cp.hdr = hdr;
        cp.states_only = 1;
        cp.dynamic = 1;
        cp.first_done = &hdr->first_done;
        const int n_prefix = kv->num_kv_heads * q_tiles * nsplit;
        const int g1 = std::min(dev->sms, n_prefix);
        LongParams c1 = cp;
        c1.wait_start = 1;
        c1.first_ctas = -1;
        rc = launch_long(c1, maps.q, *ptk, *ptv, D, g1, s);
        if (rc != PA_OK) return fail(rc, "prefix kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
        sp.no_start_wait = 1;
        sp.test_stall = 0;
        sp.out_f32 = casc->suffix_o;
        sp.lse = casc->suffix_lse;
        rc = launch_short(sp, maps.k, maps.v, D, fp8, short_grid, s);
        if (rc != PA_OK) return fail(rc, "split-KV kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
        LongParams c2 = cp;
        c2.overlap_prev = 1;
        c2.first_ctas = g1;
        rc = launch_long(c2, maps.q, *ptk, *ptv, D, n_prefix, s);
        if (rc != PA_OK) return fail(rc, "prefix kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
        PrefixFoldParams f{};
        f.partial_o = casc->prefix_o;
        f.partial_lse = casc->prefix_lse;
        f.extra_o = casc->suffix_o;
        f.extra_lse = casc->suffix_lse;
        f.nsplit = nsplit;
        f.q_tiles = q_tiles;
        f.pairs = kv->num_kv_heads * q_tiles;
        f.group = group;
        f.q_tile_tokens = tq;
        f.num_q_tokens = T;
        f.num_q_heads = Hq;
        f.out = static_cast<__nv_bfloat16 *>(out);
        f.out_f32 = nullptr;
        f.lse = lse;
        rc = launch_prefix_fold(f, D, s);
        return rc == PA_OK ? PA_OK : fail(rc, "cascade fold launch failed");
    }

    // a long request has q_len * group > short_max_rows, so there are at
    // most T / (short_max_rows / group + 1) of them
    const int min_long_tokens = short_max_rows / group + 1;
    const int max_long_reqs =
        forbid_long ? 0 : std::min(num_seqs, T / std::max(1, min_long_tokens));
    LongParams lp{};
    int long_grid = 0;
    if (max_long_reqs > 0) {
        lp.out = sp.out;
        lp.lse = lse;
        lp.out_f32 = nullptr;
        lp.block_tables = block_tables;
        lp.bt_stride = max_blocks;
        lp.qsl = qsl;
        lp.ctx = ctx;
        lp.seq_lens = seq_lens;
        lp.num_q_tokens = T;
        lp.num_q_heads = Hq;
        lp.num_kv_heads = kv->num_kv_heads;
        lp.group = group;
        lp.q_tile_tokens = tq;
        lp.block_size = kv->block_size;
        lp.num_blocks = kv->num_blocks;
        lp.kv_rows = sp.kv_rows;
        lp.scale_log2 = sp.scale_log2;
        lp.prefix_mode = 0;
        lp.hdr = hdr;
        lp.items = pp.long_items;
        lp.partial_o = sp.partial_o;
        lp.partial_lse = sp.partial_lse;
        lp.status = dev->status;
        lp.tile_counter = reinterpret_cast<unsigned long long *>(
            g_tile_counter.load(std::memory_order_relaxed));
        if (staged) {
            lp.stage_base = pp.stage_base;
            lp.k_scale = kv->k_scale;
            lp.v_scale = kv->v_scale;
            lp.num_blocks = stg.cap;
            lp.kv_rows = stg.cap * kv->num_kv_heads * kv->block_size;
        }
        long_grid = std::min(kv->num_kv_heads * ((T + tq - 1) / tq + max_long_reqs), L.max_long);
    }
    const CUtensorMap &lk = staged ? stg.tk : maps.k;
    const CUtensorMap &lv = staged ? stg.tv : maps.v;

    if (max_long_reqs > 0 && T >= kSideBySideMinTokens && !profiling_active()) {
        // The HBM-bound split-KV kernel and the tensor-core kernel run side by
        // side: a first tensor-core grid takes part of the SMs (it waits
        // for the plan, then lets the next grid in), the split-KV grid fills
        // the others, and a second tensor-core grid takes SMs over as
        // split-KV CTAs finish.  Both tensor-core grids pull items, longest
        // first, from the step's counter; the second completes only after
        // the first and after the split-KV grid.  A step of few tokens has
        // little or no tensor-core work: there the two extra launches would
        // only add latency, and the kernels run one after the other.
        LongParams l1 = lp;
        l1.dynamic = 1;
        l1.wait_start = 1;
        l1.first_done = &hdr->first_done;
        l1.first_ctas = -1;
        // share of the SMs measured best on the mixed step: two fifths beside
        // the HBM-bound bf16 split-KV kernel (60 of 152 SMs: 767.9 us per step,
        // against 769.6 with 56, 773.4 with 64 and 785.4 with 50); a tenth
        // beside the fp8 one, whose rate follows its SM count (707.3 us, 710.1
        // with an eighth)
        const int g1 = std::min(std::max(1, fp8 ? dev->sms / 10 : dev->sms * 2 / 5), long_grid);
        rc = launch_long(l1, maps.q, lk, lv, D, g1, s);
        if (rc != PA_OK) return fail(rc, "tensor-core kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
        sp.no_start_wait = 1;
        sp.claim_ahead = 0;
        sp.test_stall = 0;
        rc = launch_short(sp, maps.k, maps.v, D, fp8, short_grid, s);
        if (rc != PA_OK) return fail(rc, "split-KV kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
        LongParams l2 = lp;
        l2.dynamic = 1;
        l2.overlap_prev = 1;
        l2.first_done = &hdr->first_done;
        // the test hook waits for one CTA that the first grid never had
        l2.first_ctas = g1 + (stall == PA_TEST_STALL_LAST_GRID ? 1 : 0);
        rc = launch_long(l2, maps.q, lk, lv, D, long_grid, s);
        if (rc != PA_OK) return fail(rc, "tensor-core kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
        return PA_OK;
    }

    {
        ProfScope prof(PA_KERNEL_SPLIT_KV, s);
        rc = launch_short(sp, maps.k, maps.v, D, fp8, short_grid, s);
    }
    if (rc != PA_OK) return fail(rc, "split-KV kernel launch failed: %s",
                                 cudaGetErrorString(cudaGetLastError()));
    if (max_long_reqs > 0) {
        // the split-KV kernel was launched just before: the tensor-core grid
        // may take over SMs as split-KV CTAs finish (its rows are disjoint)
        lp.overlap_prev = short_grid > 0 ? 1 : 0;
        {
            ProfScope prof(PA_KERNEL_TENSOR_CORE, s);
            rc = launch_long(lp, maps.q, lk, lv, D, long_grid, s);
        }
        if (rc != PA_OK) return fail(rc, "tensor-core kernel launch failed: %s",
                                     cudaGetErrorString(cudaGetLastError()));
    }
    return PA_OK;
}

int common_checks(const void *q, const pa_kv_desc *kv, int32_t num_q_tokens, int32_t num_q_heads,
                  float scale, const void *out, const void *workspace) {
    int rc = check_kv(kv);
    if (rc != PA_OK) return rc;
    rc = check_heads(kv, num_q_heads);
    if (rc != PA_OK) return rc;
    if (num_q_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_q_tokens < 0");
    if (num_q_tokens > 0 && (!q || !out)) return fail(PA_ERR_INVALID_ARG, "q or out is NULL");
    if (!aligned(q, 16) || !aligned(out, 16))
        return fail(PA_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale is not finite");
    if (kv->kv_dtype == PA_KV_FP8_E4M3 && num_q_heads / kv->num_kv_heads > kShortMaxRows)
        return fail(PA_ERR_UNSUPPORTED, "fp8 KV pool: group size above %d not built",
                    kShortMaxRows);
    if (workspace && !aligned(workspace, 256))
        return fail(PA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    return PA_OK;
}

int run_prefix(const void *q, const pa_kv_desc *kv, const int32_t *prefix_blocks, int32_t prefix_len,
               int32_t T, int32_t Hq, float scale, void *out, float *lse, uint8_t *ws,
               const WsLayout &L, const StepMaps &maps, const PrefixStage &ps, DeviceInfo *dev,
               cudaStream_t s) {
    const int group = Hq / kv->num_kv_heads;
    int q_tiles, nsplit, split_keys;
    prefix_plan(T, prefix_len, kv->num_kv_heads, group, dev->sms, &q_tiles, &nsplit, &split_keys);
    // a split prefix leaves its split states to the fold kernel, which runs
    // the fold of a (kv head, query tile) on many SMs
    LongParams lp = prefix_params(kv, prefix_blocks, prefix_len, T, Hq, scale, q_tiles, nsplit,
                                  split_keys, reinterpret_cast<float *>(ws + L.prefix_o),
                                  reinterpret_cast<float *>(ws + L.prefix_lse), dev);
    lp.out = static_cast<__nv_bfloat16 *>(out);
    lp.lse = lse;
    const CUtensorMap *tk = &maps.k, *tv = &maps.v;
    int rc = stage_prefix(ps, kv, prefix_blocks, &lp, &tk, &tv, dev, s);
    if (rc != PA_OK) return rc;
    const int grid = kv->num_kv_heads * q_tiles * nsplit;
    rc = launch_long(lp, maps.q, *tk, *tv, kv->head_dim, grid, s);
    if (rc != PA_OK) return fail(rc, "prefix kernel launch failed");
    if (nsplit > 1) {
        PrefixFoldParams f{};
        f.partial_o = lp.partial_o;
        f.partial_lse = lp.partial_lse;
        f.nsplit = nsplit;
        f.q_tiles = q_tiles;
        f.pairs = kv->num_kv_heads * q_tiles;
        f.group = group;
        f.q_tile_tokens = lp.q_tile_tokens;
        f.num_q_tokens = T;
        f.num_q_heads = Hq;
        f.out = static_cast<__nv_bfloat16 *>(out);
        f.lse = lse;
        rc = launch_prefix_fold(f, kv->head_dim, s);
        if (rc != PA_OK) return fail(rc, "prefix fold launch failed");
    }
    return PA_OK;
}

int prefix_partial_rows(int T, int prefix_len, int num_kv_heads, int group) {
    int q_tiles, nsplit, split_keys;
    // the split count never exceeds 64, whatever the SM count
    prefix_plan(T, prefix_len, num_kv_heads, group, 1 << 20, &q_tiles, &nsplit, &split_keys);
    return num_kv_heads * q_tiles * nsplit * kLongRows;
}

}  // namespace

namespace pa {

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Attention for one step inside a caller-provided scratch region of fixed
// size (used by the entry point that never allocates).  The work lists get
// the smallest capacity that always fits (one split per request and kv
// head, plus room for extra splits); whatever space is left holds split-KV
// partial states, and the planner picks split sizes that fit it.
int attention_in_fixed_workspace(const void *q, const pa_kv_desc *kv,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *query_start_loc, const int32_t *context_lens,
                                 const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_tokens,
                                 int32_t num_q_heads, float scale, void *out, float *lse,
                                 void *scratch, size_t scratch_bytes, cudaStream_t s) {
    g_err[0] = 0;
    int rc = common_checks(q, kv, num_q_tokens, num_q_heads, scale, out, scratch);
    if (rc != PA_OK) return rc;
    if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (num_seqs == 0 || num_q_tokens == 0) return PA_OK;
    if (!block_tables || !query_start_loc || !context_lens || !seq_lens)
        return fail(PA_ERR_INVALID_ARG, "metadata pointer is NULL");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq <= 0");
    const int hkv = kv->num_kv_heads, D = kv->head_dim;
    const int tq = q_tile_tokens(num_q_heads / hkv);
    WsLayout L{};
    const int pieces = pieces_bound(num_seqs, num_q_tokens, num_q_heads / hkv);
    L.max_short = hkv * pieces + 4096;
    L.max_long = hkv * ((num_q_tokens + tq - 1) / tq + num_seqs);
    L.num_counters = hkv * pieces;
    size_t off = 0;
    L.header = off;
    off = align256(off + sizeof(PlanHeader));
    L.counters = off;
    off = align256(off + sizeof(int) * static_cast<size_t>(L.num_counters));
    L.short_items = off;
    off = align256(off + sizeof(ShortItem) * static_cast<size_t>(L.max_short));
    L.long_items = off;
    off = align256(off + sizeof(LongItem) * static_cast<size_t>(L.max_long));
    const size_t fixed = off + 512;  // + alignment of the two partial arrays
    if (fixed > scratch_bytes)
        return fail(PA_ERR_WORKSPACE,
                    "step too large for the fixed scratch: its work lists need %zu bytes, "
                    "the scratch holds %zu", fixed, scratch_bytes);
    const size_t rows = (scratch_bytes - fixed) / (sizeof(float) * (static_cast<size_t>(D) + 1));
    L.cap_rows = static_cast<int>(std::min<size_t>(rows, 1u << 24));
    L.partial_o = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(L.cap_rows) * D);
    L.partial_lse = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(L.cap_rows));
    L.total = off;
    if (L.total > scratch_bytes) return fail(PA_ERR_WORKSPACE, "scratch layout overflow");
    DeviceInfo *dev;
    if ((rc = device_info(&dev)) != PA_OK) return rc;
    StepMaps maps;
    if ((rc = make_maps(&maps, q, kv, num_q_tokens, num_q_heads)) != PA_OK) return rc;
    return run_step(q, kv, block_tables, max_blocks_per_seq, query_start_loc, context_lens,
                    seq_lens, num_seqs, num_q_tokens, num_q_heads, scale, out, lse,
                    static_cast<uint8_t *>(scratch), L, kShortMaxRows, 0, nullptr, false, maps,
                    Staging(), dev, s);
}

int set_error_message(int code, const char *msg) { return fail(code, "%s", msg); }

}  // namespace pa

extern "C" {

const char *pa_last_error_message(void) { return g_err; }

const char *pa_status_string(int code) {
    switch (code) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_BAD_METADATA: return "PA_ERR_BAD_METADATA";
    default: return "PA_ERR_UNKNOWN";
    }
}

int pa_write_kv(const void *k, const void *v, const int64_t *slot_mapping, int32_t num_tokens,
                const pa_kv_desc *kv, void *stream) {
    g_err[0] = 0;
    int rc = check_kv(kv);
    if (rc != PA_OK) return rc;
    if ((rc = check_new_rows(NewRows{k, v, slot_mapping, num_tokens})) != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    DeviceInfo *dev;
    if ((rc = device_info(&dev)) != PA_OK) return rc;
    {
        ProfScope prof(PA_KERNEL_WRITE_KV, static_cast<cudaStream_t>(stream));
        rc = launch_write_kv(k, v, slot_mapping, num_tokens, kv, dev->status,
                             static_cast<cudaStream_t>(stream));
    }
    return rc == PA_OK ? PA_OK : fail(rc, "write_kv launch failed");
}

size_t pa_attention_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim) {
    if (num_seqs < 0 || num_q_tokens < 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || (head_dim != 64 && head_dim != 128))
        return 0;
    return make_layout(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, 0, false).total;
}

}  // extern "C"

namespace {

// pa_attention_ex, and with `fresh` the write of the step's new rows first.
int attention_entry(const void *q, const pa_kv_desc *kv, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                    const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                    int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out, float *lse,
                    void *workspace, size_t workspace_bytes, int32_t short_q_max_rows,
                    int32_t split_keys, cudaStream_t stream, const NewRows *fresh) {
    g_err[0] = 0;
    int rc = common_checks(q, kv, num_q_tokens, num_q_heads, scale, out, workspace);
    if (rc != PA_OK) return rc;
    if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (short_q_max_rows < -1 || short_q_max_rows > kShortMaxRows)
        return fail(PA_ERR_INVALID_ARG, "short_q_max_rows must be -1 or in [0, %d]", kShortMaxRows);
    if (split_keys < 0 || split_keys % kStageKeys != 0)
        return fail(PA_ERR_INVALID_ARG, "split_keys must be 0 or a multiple of %d", kStageKeys);
    if (fresh && (rc = check_new_rows(*fresh)) != PA_OK) return rc;
    if (num_seqs == 0 || num_q_tokens == 0) {
        // nothing to attend: the write alone, as pa_write_kv
        if (!fresh || fresh->num_tokens == 0) return PA_OK;
        DeviceInfo *dev;
        if ((rc = device_info(&dev)) != PA_OK) return rc;
        ProfScope prof(PA_KERNEL_WRITE_KV, stream);
        rc = launch_write_kv(fresh->k, fresh->v, fresh->slots, fresh->num_tokens, kv, dev->status,
                             stream);
        return rc == PA_OK ? PA_OK : fail(rc, "write_kv launch failed");
    }
    if (!block_tables || !query_start_loc || !context_lens || !seq_lens)
        return fail(PA_ERR_INVALID_ARG, "metadata pointer is NULL");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq <= 0");
    const WsLayout L = make_layout(num_seqs, num_q_tokens, num_q_heads, kv->num_kv_heads,
                                   kv->head_dim, 0, false);
    if (!workspace || workspace_bytes < L.total)
        return fail(PA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", L.total,
                    workspace_bytes);
    DeviceInfo *dev;
    if ((rc = device_info(&dev)) != PA_OK) return rc;
    StepMaps maps;
    if ((rc = make_maps(&maps, q, kv, num_q_tokens, num_q_heads)) != PA_OK) return rc;
    // an fp8 pool stages long requests in the workspace beyond the layout
    Staging stg;
    if ((rc = make_staging(&stg, kv, static_cast<uint8_t *>(workspace), L.total, workspace_bytes)) !=
        PA_OK)
        return rc;
    return run_step(q, kv, block_tables, max_blocks_per_seq, query_start_loc, context_lens,
                    seq_lens, num_seqs, num_q_tokens, num_q_heads, scale, out, lse,
                    static_cast<uint8_t *>(workspace), L,
                    short_q_max_rows < 0 ? kShortMaxRows : short_q_max_rows, split_keys, nullptr,
                    false, maps, stg, dev, stream, fresh);
}

}  // namespace

extern "C" {

int pa_attention_ex(const void *q, const pa_kv_desc *kv, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                    const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                    int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out, float *lse,
                    void *workspace, size_t workspace_bytes, int32_t short_q_max_rows,
                    int32_t split_keys, void *stream) {
    return attention_entry(q, kv, block_tables, max_blocks_per_seq, query_start_loc,
                               context_lens, seq_lens, num_seqs, num_q_tokens, num_q_heads, scale,
                               out, lse, workspace, workspace_bytes, short_q_max_rows, split_keys,
                               static_cast<cudaStream_t>(stream), nullptr);
}

int pa_write_kv_attention(const void *k, const void *v, const int64_t *slot_mapping,
                          int32_t num_new_tokens, const void *q, const pa_kv_desc *kv,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *query_start_loc, const int32_t *context_lens,
                          const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_tokens,
                          int32_t num_q_heads, float scale, void *out, float *lse,
                          void *workspace, size_t workspace_bytes, void *stream) {
    const NewRows fresh{k, v, slot_mapping, num_new_tokens};
    return attention_entry(q, kv, block_tables, max_blocks_per_seq, query_start_loc,
                               context_lens, seq_lens, num_seqs, num_q_tokens, num_q_heads, scale,
                               out, lse, workspace, workspace_bytes, -1, 0,
                               static_cast<cudaStream_t>(stream), &fresh);
}



size_t pa_fp8_staging_bytes(int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int64_t num_blocks) {
    if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0) return 0;
    const size_t blk = static_cast<size_t>(num_kv_heads) * block_size * head_dim * 2;
    return 2 * align256(static_cast<size_t>(num_blocks) * blk) + 768;
}

int pa_attention(const void *q, const pa_kv_desc *kv, const int32_t *block_tables,
                 int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                 const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                 int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out, float *lse,
                 void *workspace, size_t workspace_bytes, void *stream) {
    return pa_attention_ex(q, kv, block_tables, max_blocks_per_seq, query_start_loc, context_lens,
                           seq_lens, num_seqs, num_q_tokens, num_q_heads, scale, out, lse,
                           workspace, workspace_bytes, -1, 0, stream);
}

int pa_merge_states(const void *o_a, const float *lse_a, const void *o_b, const float *lse_b,
                    int32_t n, int32_t num_heads, int32_t head_dim, void *out, float *lse_out,
                    void *stream) {
    g_err[0] = 0;
    if (n < 0 || num_heads <= 0) return fail(PA_ERR_INVALID_ARG, "bad n / num_heads");
    if (head_dim <= 0 || head_dim % 8 != 0)
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be a positive multiple of 8");
    if (n == 0) return PA_OK;
    if (!o_a || !o_b || !lse_a || !lse_b || !out) return fail(PA_ERR_INVALID_ARG, "NULL input");
    if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(out, 16))
        return fail(PA_ERR_INVALID_ARG, "o_a, o_b and out must be 16-byte aligned");
    const int rc = launch_merge(o_a, lse_a, o_b, lse_b, n, num_heads, head_dim, out, lse_out,
                                static_cast<cudaStream_t>(stream));
    return rc == PA_OK ? PA_OK : fail(rc, "merge launch failed");
}

size_t pa_cascade_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t prefix_len) {
    if (num_seqs < 0 || num_q_tokens < 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || (head_dim != 64 && head_dim != 128) || prefix_len < 0)
        return 0;
    const int group = num_q_heads / num_kv_heads;
    const int rows = prefix_partial_rows(num_q_tokens, prefix_len, num_kv_heads, group);
    return make_layout(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, rows, true)
        .total;
}

int pa_prefix_attention(const void *q, const pa_kv_desc *kv, const int32_t *prefix_blocks,
                        int32_t prefix_len, int32_t num_q_tokens, int32_t num_q_heads,
                        float scale, void *out, float *lse, void *workspace,
                        size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = common_checks(q, kv, num_q_tokens, num_q_heads, scale, out, workspace);
    if (rc != PA_OK) return rc;
    if (prefix_len < 0) return fail(PA_ERR_INVALID_ARG, "prefix_len < 0");
    if (prefix_len > 0 && !prefix_blocks) return fail(PA_ERR_INVALID_ARG, "prefix_blocks is NULL");
    if (num_q_tokens == 0) return PA_OK;
    const int group = num_q_heads / kv->num_kv_heads;
    const WsLayout L = make_layout(1, num_q_tokens, num_q_heads, kv->num_kv_heads, kv->head_dim,
                                   prefix_partial_rows(num_q_tokens, prefix_len, kv->num_kv_heads,
                                                       group),
                                   true);
    if (!workspace || workspace_bytes < L.total)
        return fail(PA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", L.total,
                    workspace_bytes);
    PrefixStage ps;
    if ((rc = make_prefix_stage(&ps, kv, prefix_len, static_cast<uint8_t *>(workspace), L.total,
                                workspace_bytes)) != PA_OK)
        return rc;
    DeviceInfo *dev;
    if ((rc = device_info(&dev)) != PA_OK) return rc;
    StepMaps maps;
    if ((rc = make_maps(&maps, q, kv, num_q_tokens, num_q_heads)) != PA_OK) return rc;
    return run_prefix(q, kv, prefix_blocks, prefix_len, num_q_tokens, num_q_heads, scale, out,
                      lse, static_cast<uint8_t *>(workspace), L, maps, ps, dev,
                      static_cast<cudaStream_t>(stream));
}

int pa_cascade_decode(const void *q, const pa_kv_desc *kv, const int32_t *prefix_blocks,
                      int32_t prefix_len, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                      const int32_t *context_lens, const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_q_tokens, int32_t num_q_heads, float scale, void *out,
                      float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    int rc = common_checks(q, kv, num_q_tokens, num_q_heads, scale, out, workspace);
    if (rc != PA_OK) return rc;
    if (num_q_heads / kv->num_kv_heads > kShortMaxRows)
        return fail(PA_ERR_UNSUPPORTED, "cascade decode: group size above %d not built",
                    kShortMaxRows);
    if (num_seqs < 0 || prefix_len < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (prefix_len > 0 && !prefix_blocks) return fail(PA_ERR_INVALID_ARG, "prefix_blocks is NULL");
    if (num_seqs == 0 || num_q_tokens == 0) return PA_OK;
    if (!block_tables || !query_start_loc || !context_lens || !seq_lens)
        return fail(PA_ERR_INVALID_ARG, "metadata pointer is NULL");
    if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq <= 0");
    const int group = num_q_heads / kv->num_kv_heads;
    const WsLayout L = make_layout(num_seqs, num_q_tokens, num_q_heads, kv->num_kv_heads,
                                   kv->head_dim,
                                   prefix_partial_rows(num_q_tokens, prefix_len, kv->num_kv_heads,
                                                       group),
                                   true);
    if (!workspace || workspace_bytes < L.total)
        return fail(PA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", L.total,
                    workspace_bytes);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    PrefixStage ps;
    if ((rc = make_prefix_stage(&ps, kv, prefix_len, ws, L.total, workspace_bytes)) != PA_OK)
        return rc;
    DeviceInfo *dev;
    if ((rc = device_info(&dev)) != PA_OK) return rc;
    StepMaps maps;
    if ((rc = make_maps(&maps, q, kv, num_q_tokens, num_q_heads)) != PA_OK) return rc;
    CascadeArgs casc;
    casc.prefix_blocks = prefix_blocks;
    casc.prefix_len = prefix_len;
    casc.ps = &ps;
    casc.prefix_o = reinterpret_cast<float *>(ws + L.prefix_o);
    casc.prefix_lse = reinterpret_cast<float *>(ws + L.prefix_lse);
    casc.suffix_o = reinterpret_cast<float *>(ws + L.extra_o);
    casc.suffix_lse = reinterpret_cast<float *>(ws + L.extra_lse);
    return run_step(q, kv, block_tables, max_blocks_per_seq, query_start_loc, context_lens,
                    seq_lens, num_seqs, num_q_tokens, num_q_heads, scale, out, lse, ws, L,
                    kShortMaxRows, 0, &casc, true, maps, Staging(), dev,
                    static_cast<cudaStream_t>(stream));
}

size_t pa_cascade_fp8_staging_bytes(int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t prefix_len) {
    if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || prefix_len < 0) return 0;
    return prefix_stage_bytes(num_kv_heads, head_dim, block_size, prefix_len);
}

int pa_validate_metadata(const int32_t *block_tables, int32_t max_blocks_per_seq,
                         const int32_t *query_start_loc, const int32_t *context_lens,
                         const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_tokens,
                         const int64_t *slot_mapping, int32_t num_blocks, int32_t block_size) {
    g_err[0] = 0;
    if (num_seqs < 0 || num_q_tokens < 0 || block_size <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad sizes");
    if (num_seqs > 0 && (!block_tables || !query_start_loc || !context_lens || !seq_lens))
        return fail(PA_ERR_INVALID_ARG, "metadata pointer is NULL");
    if (num_seqs > 0 && query_start_loc[0] != 0)
        return fail(PA_ERR_BAD_METADATA, "query_start_loc[0] = %d, expected 0", query_start_loc[0]);
    for (int b = 0; b < num_seqs; ++b) {
        const int n = query_start_loc[b + 1] - query_start_loc[b];
        if (n < 0) return fail(PA_ERR_BAD_METADATA, "query_start_loc decreases at %d", b);
        if (context_lens[b] < 0) return fail(PA_ERR_BAD_METADATA, "context_lens[%d] < 0", b);
        if (seq_lens[b] != context_lens[b] + n)
            return fail(PA_ERR_BAD_METADATA, "seq_lens[%d]=%d != context %d + q_len %d", b,
                        seq_lens[b], context_lens[b], n);
        const int64_t nblk = (static_cast<int64_t>(seq_lens[b]) + block_size - 1) / block_size;
        if (nblk > max_blocks_per_seq)
            return fail(PA_ERR_BAD_METADATA, "request %d needs %lld blocks > max_blocks_per_seq",
                        b, (long long)nblk);
        for (int64_t j = 0; j < nblk; ++j) {
            const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + j];
            if (blk < 0 || blk >= num_blocks)
                return fail(PA_ERR_BAD_METADATA, "block_tables[%d][%lld] = %d out of range", b,
                            (long long)j, blk);
        }
    }
    if (num_seqs > 0 && query_start_loc[num_seqs] > num_q_tokens)
        return fail(PA_ERR_BAD_METADATA, "query_start_loc[num_seqs] = %d > num_q_tokens %d",
                    query_start_loc[num_seqs], num_q_tokens);
    if (slot_mapping && num_q_tokens > 0) {
        const int64_t nslots = static_cast<int64_t>(num_blocks) * block_size;
        // duplicates: mark slots in a bitmap
        std::vector<uint8_t> seen(static_cast<size_t>((nslots + 7) / 8), 0);
        for (int t = 0; t < num_q_tokens; ++t) {
            const int64_t s = slot_mapping[t];
            if (s < 0) continue;
            if (s >= nslots) return fail(PA_ERR_BAD_METADATA, "slot_mapping[%d] = %lld outside pool", t, (long long)s);
            uint8_t &byte = seen[static_cast<size_t>(s >> 3)];
            const uint8_t bit = static_cast<uint8_t>(1u << (s & 7));
            if (byte & bit) return fail(PA_ERR_BAD_METADATA, "slot %lld used twice", (long long)s);
            byte |= bit;
        }
    }
    return PA_OK;
}

int pa_set_profile_events(int32_t which, void *start_event, void *end_event) {
    g_err[0] = 0;
    if (which < 0 || which > 3) return fail(PA_ERR_INVALID_ARG, "unknown kernel id %d", which);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof[which][0] = start_event;
    g_prof[which][1] = end_event;
    return PA_OK;
}

int pa_set_tile_counter(uint64_t *counter) {
    g_err[0] = 0;
    if (counter && !aligned(counter, 8))
        return fail(PA_ERR_INVALID_ARG, "tile counter must be 8-byte aligned");
    g_tile_counter.store(counter, std::memory_order_relaxed);
    return PA_OK;
}

int pa_set_test_stall(int32_t which) {
    g_err[0] = 0;
    if (which != PA_TEST_STALL_NONE && which != PA_TEST_STALL_SPLIT_KV &&
        which != PA_TEST_STALL_LAST_GRID)
        return fail(PA_ERR_INVALID_ARG, "unknown test stall %d", which);
    g_test_stall.store(which, std::memory_order_relaxed);
    return PA_OK;
}

int pa_read_device_status(uint32_t *status, int clear, void *stream) {
    g_err[0] = 0;
    if (!status) return fail(PA_ERR_INVALID_ARG, "status is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return fail(PA_ERR_CUDA, "stream sync failed");
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pa_status, sizeof v) != cudaSuccess)
        return fail(PA_ERR_CUDA, "status read failed");
    *status = v;
    if (clear) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_pa_status, &zero, sizeof zero) != cudaSuccess)
            return fail(PA_ERR_CUDA, "status clear failed");
    }
    return PA_OK;
}

uint64_t pa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
