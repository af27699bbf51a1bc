// pa_static.cu -- paged attention that never allocates device memory.
//
// pa_attention needs a workspace for its device-built work list, split-KV
// partial states and completion counters, and the caller normally allocates
// it.  Some callers cannot: a host runtime whose device memory is handed out
// only at start-up (a fixed arena, nothing can be added later), code that
// runs where allocation is forbidden or unsafe (a memory-pressure or shutdown
// path of a serving engine, or a plugin that must not create device buffers
// of its own).  This entry point serves them: its scratch is one fixed array
// in the library's own device memory, so a call only needs the inputs and
// outputs.
//
// Costs and rules for users:
//  * this file is its own device module, and under lazy module loading (the
//    CUDA default) a module is loaded on a device when the library first
//    needs it there: the array's PA_NO_ALLOC_SCRATCH_BYTES are committed on a
//    device at the first call of this entry point on that device (which looks
//    up the array's address), and held until the process exits.  A caller
//    that must not allocate later should make one call at start-up on every
//    device it will use -- that first call can fail with PA_ERR_CUDA if the
//    device has no room left -- and before any stream capture begins;
//  * all calls on a device share the one array and it keeps the last call's
//    contents: calls whose kernels overlap on the GPU (other streams, other
//    host threads) race on it and give wrong results -- order them;
//  * a step whose work lists do not fit the array is refused with
//    PA_ERR_WORKSPACE and a message.  The work lists get the smallest room
//    that always fits one split per request piece and kv head, and the
//    partial-state area whatever is left, so a large batch may be given
//    longer (fewer) splits than pa_attention would choose -- same results,
//    up to rounding;
//  * on an fp8 (e4m3) pool there is no room for the bf16 staging copy the
//    tensor-core path reads, so every request (long ones in pieces of
//    64 / group query tokens) runs on the split-KV kernel.
#include <mutex>

#include "pa_internal.cuh"

static __device__ __align__(256) unsigned char g_no_alloc_scratch[PA_NO_ALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;
}  // namespace

extern "C" int pa_attention_no_alloc(const void *q, const pa_kv_desc *kv,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *query_start_loc, const int32_t *context_lens,
                                     const int32_t *seq_lens, int32_t num_seqs,
                                     int32_t num_q_tokens, int32_t num_q_heads, float scale,
                                     void *out, float *lse, void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return pa::set_error_message(PA_ERR_CUDA, "no current CUDA device");
    void *scratch = nullptr;
    {
        // One-time set-up per device, with that device current: the host
        // name of the array is not a device address; ask the runtime for it.
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_addr[dev]) {
            void *p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
            if (e != cudaSuccess || !p)
                return pa::set_error_message(PA_ERR_CUDA,
                                             "cudaGetSymbolAddress of the no-alloc scratch failed");
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    return pa::attention_in_fixed_workspace(q, kv, block_tables, max_blocks_per_seq,
                                            query_start_loc, context_lens, seq_lens, num_seqs,
                                            num_q_tokens, num_q_heads, scale, out, lse, scratch,
                                            PA_NO_ALLOC_SCRATCH_BYTES,
                                            static_cast<cudaStream_t>(stream));
}
