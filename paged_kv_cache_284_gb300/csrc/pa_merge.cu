// pa_merge.cu -- the merge operator of cascade inference (2048ai.net page on
// the vLLM V1 engine, §02 推理优化 › 1. 级联推理): two attention states over
// disjoint key sets, (o_a, lse_a) and (o_b, lse_b), combine into the state
// over the union:
//   M = max(lse_a, lse_b), lse = M + ln(e^(lse_a-M) + e^(lse_b-M)),
//   o = e^(lse_a-lse) o_a + e^(lse_b-lse) o_b.
// HBM-bound elementwise kernel: one thread per 8 output elements (16 bytes
// of bf16), fp32 arithmetic.
#include "pa_internal.cuh"

namespace pa {

__global__ void __launch_bounds__(256) merge_states_kernel(
    const uint4 *__restrict__ oa, const float *__restrict__ la, const uint4 *__restrict__ ob,
    const float *__restrict__ lb, int64_t rows, int pieces_per_row, uint4 *__restrict__ out,
    float *__restrict__ lse_out) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= rows * pieces_per_row) return;
    const int64_t row = idx / pieces_per_row;
    const float a = __ldg(la + row), b = __ldg(lb + row);
    const float m = fmaxf(a, b);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (m != -INFINITY) {
        const float ea = __expf(a - m), eb = __expf(b - m);
        const float inv = 1.f / (ea + eb);
        wa = ea * inv;
        wb = eb * inv;
        l = m + __logf(ea + eb);
    }
    const uint4 va = __ldg(oa + idx), vb = __ldg(ob + idx);
    const __nv_bfloat162 *pa2 = reinterpret_cast<const __nv_bfloat162 *>(&va);
    const __nv_bfloat162 *pb2 = reinterpret_cast<const __nv_bfloat162 *>(&vb);
    uint4 res;
    uint32_t *pr = reinterpret_cast<uint32_t *>(&res);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(pa2[i]);
        const float2 fb = __bfloat1622float2(pb2[i]);
        pr[i] = pack_bf16x2(wa * fa.x + wb * fb.x, wa * fa.y + wb * fb.y);
    }
    out[idx] = res;
    if (lse_out && (idx - row * pieces_per_row) == 0) lse_out[row] = l;
}

int launch_merge(const void *oa, const float *la, const void *ob, const float *lb, int n,
                 int heads, int head_dim, void *out, float *lse_out, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(n) * heads;
    if (rows == 0) return PA_OK;
    const int pieces = head_dim / 8;
    const int64_t total = rows * pieces;
    const int threads = 256;
    PdlLaunch l(static_cast<unsigned>((total + threads - 1) / threads), threads, 0, s, false);
    return launch_kernel(l, merge_states_kernel, static_cast<const uint4 *>(oa), la,
                         static_cast<const uint4 *>(ob), lb, rows, pieces,
                         static_cast<uint4 *>(out), lse_out) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

}  // namespace pa
