// pa_static.cu -- paged attention that never allocates device memory.
//
// pa_attention needs a workspace for its device-built work list, split-KV
// partial states and completion counters, and the caller normally allocates
// it.  Some callers cannot: a host runtime whose device memory is handed out
// only at start-up (a fixed arena, nothing can be added later), code that
// runs where allocation is forbidden or unsafe (a memory-pressure or shutdown
// path of a serving engine, or a plugin that must not create device buffers
// of its own).  This entry point serves them: its scratch is one fixed array
// in the library's own device memory, created when the library is loaded on a
// device, so a call only needs the inputs and outputs.
//
// Costs and rules for users:
//  * every GPU that loads the library holds PA_NO_ALLOC_SCRATCH_BYTES of device
//    memory for this array until the process exits;
//  * all calls on a device share the one array and it keeps the last call's
//    contents: calls whose kernels overlap on the GPU (other streams, other
//    host threads) race on it and give wrong results -- order them;
//  * the first call on each device looks up the array's device address; make
//    that first call before any stream capture begins;
//  * a step whose work list does not fit the array is refused with
//    PA_ERR_WORKSPACE and a message; smaller split-KV partial space only makes
//    the planner choose longer splits.
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
