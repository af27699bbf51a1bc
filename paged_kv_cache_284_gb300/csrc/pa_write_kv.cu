// pa_write_kv.cu -- reshape_and_cache: scatter this step's K/V rows into
// their cache slots (bf16 pool: bit copy; fp8 pool: quantised per kv head) ("11. 推理加速(一):vLLM 原理", §11.2: tokens fill
// fixed-size physical blocks; slot = block * block_size + offset).
//
// Pure HBM copy: each thread moves one 16-byte piece of one (token, kv head)
// row for K and the same piece for V, so a warp covers whole 16-byte sectors
// of the destination rows.
#include <algorithm>

#include <cuda_fp8.h>

#include "pa_internal.cuh"

namespace pa {

// The step's new K/V rows and their cache slots (reshape_and_cache).  A
// piece is 16 bytes of one (token, kv head) cache row: 8 bf16 elements, or
// 16 e4m3 codes quantised from 16 bf16 source elements.
struct RowWrite {
    const uint4 *k, *v;  // bf16 [num_tokens][num_kv_heads][head_dim]
    const int64_t *slots;
    uint4 *k_cache, *v_cache;
    const float *k_scale, *v_scale;  // fp8 pool only
    int num_tokens, num_kv_heads, pieces_per_row, block_size, num_blocks, fp8;
    __host__ __device__ int64_t pieces() const {
        return static_cast<int64_t>(num_tokens) * num_kv_heads * pieces_per_row;
    }
};

// Cache piece of RowWrite piece idx (< w.pieces()), or -1 for a padding
// token (negative slot) or a slot beyond the pool (flagged).
__device__ __forceinline__ int64_t row_piece_dst(const RowWrite &w, int64_t idx,
                                                 unsigned *status) {
    const int64_t per_token = static_cast<int64_t>(w.num_kv_heads) * w.pieces_per_row;
    const int64_t t = idx / per_token;
    const int64_t rem = idx - t * per_token;  // = h * pieces_per_row + piece
    const int64_t s = __ldg(w.slots + t);
    if (s < 0) return -1;
    const int64_t blk = s / w.block_size;
    const int64_t off = s - blk * w.block_size;
    if (blk >= w.num_blocks) {
        flag_status(status, PA_DEV_BAD_SLOT);
        return -1;
    }
    const int64_t h = rem / w.pieces_per_row;
    const int64_t piece = rem - h * w.pieces_per_row;
    return ((blk * w.num_kv_heads + h) * w.block_size + off) * w.pieces_per_row + piece;
}

// Four bf16 elements to four e4m3 codes: x / scale in binary32 (IEEE
// division), then the saturating round-to-nearest-even conversion.
__device__ __forceinline__ uint32_t quantise4(uint2 x, float s) {
    const float f0 = __fdiv_rn(__uint_as_float(x.x << 16), s);
    const float f1 = __fdiv_rn(__uint_as_float(x.x & 0xFFFF0000u), s);
    const float f2 = __fdiv_rn(__uint_as_float(x.y << 16), s);
    const float f3 = __fdiv_rn(__uint_as_float(x.y & 0xFFFF0000u), s);
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f0, f1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f2, f3), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi << 16);
}
__device__ __forceinline__ uint4 quantise16(uint4 a, uint4 b, float s) {
    return make_uint4(quantise4(make_uint2(a.x, a.y), s), quantise4(make_uint2(a.z, a.w), s),
                      quantise4(make_uint2(b.x, b.y), s), quantise4(make_uint2(b.z, b.w), s));
}

// Writes K and V piece idx (< w.pieces()) of the new rows into a bf16
// pool's cache: a bit copy.
__device__ __forceinline__ void write_row_piece_bf16(const RowWrite &w, int64_t idx,
                                                     unsigned *status) {
    const int64_t dst = row_piece_dst(w, idx, status);
    if (dst < 0) return;
    const uint4 k = __ldg(w.k + idx), v = __ldg(w.v + idx);
    w.k_cache[dst] = k;
    w.v_cache[dst] = v;
}

// The same on an fp8 pool: the 16 bf16 source elements of the piece
// quantised with kv head h's scale.
__device__ __forceinline__ void write_row_piece_fp8(const RowWrite &w, int64_t idx,
                                                    unsigned *status) {
    const int64_t dst = row_piece_dst(w, idx, status);
    if (dst < 0) return;
    const int h = static_cast<int>((idx / w.pieces_per_row) % w.num_kv_heads);
    const float ks = __ldg(w.k_scale + h), vs = __ldg(w.v_scale + h);
    const uint4 ka = __ldg(w.k + 2 * idx), kb = __ldg(w.k + 2 * idx + 1);
    const uint4 va = __ldg(w.v + 2 * idx), vb = __ldg(w.v + 2 * idx + 1);
    w.k_cache[dst] = quantise16(ka, kb, ks);
    w.v_cache[dst] = quantise16(va, vb, vs);
}

static RowWrite make_row_write(const void *k, const void *v, const int64_t *slots,
                               int num_tokens, const pa_kv_desc *kv) {
    RowWrite w{};
    w.k = static_cast<const uint4 *>(k);
    w.v = static_cast<const uint4 *>(v);
    w.slots = slots;
    w.k_cache = static_cast<uint4 *>(kv->k_cache);
    w.v_cache = static_cast<uint4 *>(kv->v_cache);
    w.fp8 = kv->kv_dtype == PA_KV_FP8_E4M3 ? 1 : 0;
    w.k_scale = w.fp8 ? kv->k_scale : nullptr;
    w.v_scale = w.fp8 ? kv->v_scale : nullptr;
    w.num_tokens = num_tokens;
    w.num_kv_heads = kv->num_kv_heads;
    // a 16-byte cache piece holds 8 bf16 elements or 16 e4m3 codes
    w.pieces_per_row = w.fp8 ? kv->head_dim / 16 : kv->head_dim / 8;
    w.block_size = kv->block_size;
    w.num_blocks = kv->num_blocks;
    return w;
}

template <bool FP8>
__global__ void __launch_bounds__(256) write_kv_kernel(const RowWrite w, unsigned *status) {
    // k, v and the slots may come from the previous kernel, and that kernel
    // may still read the cache
    pdl_wait();
    pdl_trigger();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= w.pieces()) return;
    if (FP8)
        write_row_piece_fp8(w, idx, status);
    else
        write_row_piece_bf16(w, idx, status);
}

int launch_write_kv(const void *k, const void *v, const int64_t *slots, int num_tokens,
                    const pa_kv_desc *kv, unsigned *status, cudaStream_t s) {
    if (num_tokens == 0) return PA_OK;
    const RowWrite w = make_row_write(k, v, slots, num_tokens, kv);
    const int threads = 256;
    const int64_t blocks = (w.pieces() + threads - 1) / threads;
    PdlLaunch l(static_cast<unsigned>(blocks), threads, 0, s);
    const cudaError_t e = w.fp8 ? launch_kernel(l, write_kv_kernel<true>, w, status)
                                : launch_kernel(l, write_kv_kernel<false>, w, status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Decodes e4m3 block src of the pool into bf16 staging block k (exact: every
// e4m3 value is a bf16 value; the per-kv-head scales stay with the
// attention kernel), the block's threads striding over its 16-code pieces.
__device__ __forceinline__ void decode_block(const uint4 *__restrict__ kc8,
                                             const uint4 *__restrict__ vc8, int64_t src,
                                             int pieces_per_block, int64_t k,
                                             uint4 *__restrict__ sk, uint4 *__restrict__ sv) {
    for (int q = threadIdx.x; q < pieces_per_block; q += blockDim.x) {
        // 16 codes -> 16 bf16 (two 16-byte pieces)
        const uint4 ck = __ldg(kc8 + src * pieces_per_block + q);
        const uint4 cv = __ldg(vc8 + src * pieces_per_block + q);
        uint4 out[4];
        const uint32_t wk[4] = {ck.x, ck.y, ck.z, ck.w}, wv[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t k0, k1, v0, v1;
            e4m3x4_to_f16x2x2(wk[w], k0, k1);
            e4m3x4_to_f16x2x2(wv[w], v0, v1);
            const __half2 hk0 = *reinterpret_cast<__half2 *>(&k0), hk1 = *reinterpret_cast<__half2 *>(&k1);
            const __half2 hv0 = *reinterpret_cast<__half2 *>(&v0), hv1 = *reinterpret_cast<__half2 *>(&v1);
            const float2 fk0 = __half22float2(hk0), fk1 = __half22float2(hk1);
            const float2 fv0 = __half22float2(hv0), fv1 = __half22float2(hv1);
            // out[0..1]: K (8 bf16 each), out[2..3]: V
            reinterpret_cast<uint32_t *>(&out[w >> 1])[(w & 1) * 2] = pack_bf16x2(fk0.x, fk0.y);
            reinterpret_cast<uint32_t *>(&out[w >> 1])[(w & 1) * 2 + 1] = pack_bf16x2(fk1.x, fk1.y);
            reinterpret_cast<uint32_t *>(&out[2 + (w >> 1)])[(w & 1) * 2] = pack_bf16x2(fv0.x, fv0.y);
            reinterpret_cast<uint32_t *>(&out[2 + (w >> 1)])[(w & 1) * 2 + 1] = pack_bf16x2(fv1.x, fv1.y);
        }
        const int64_t dst = (k * pieces_per_block + q) * 2;
        sk[dst] = out[0];
        sk[dst + 1] = out[1];
        sv[dst] = out[2];
        sv[dst + 1] = out[3];
    }
}

// Staging copy of the e4m3 blocks of long requests for the tensor-core
// kernel: staging block k of staged request b (k = stage_base[b] + j) holds
// block j of b's table decoded to bf16.  Grid-stride over staging blocks;
// thread 0 finds the request of a block by binary search over the staged
// requests' first blocks.
__global__ void __launch_bounds__(256) stage_fp8_kernel(
    const uint4 *__restrict__ kc8, const uint4 *__restrict__ vc8, int num_blocks,
    int pieces_per_block, const int32_t *__restrict__ bt, int bt_stride, const PlanHeader *hdr,
    const int *stage_base, const int *stage_list, uint4 *__restrict__ sk, uint4 *__restrict__ sv,
    unsigned *status) {
    pdl_wait();  // the plan that chose the staged requests
    pdl_trigger();
    __shared__ int s_src;
    const int ns = *reinterpret_cast<const volatile int *>(&hdr->num_staged);
    const int total = *reinterpret_cast<const volatile int *>(&hdr->staged_blocks);
    for (int k = blockIdx.x; k < total; k += gridDim.x) {
        if (threadIdx.x == 0) {
            int lo = 0, hi = ns - 1;  // last staged request whose first block <= k
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldcg(stage_base + __ldcg(stage_list + mid)) <= k) lo = mid; else hi = mid - 1;
            }
            const int b = __ldcg(stage_list + lo);
            const int j = k - __ldcg(stage_base + b);
            int src = (j < bt_stride) ? __ldg(bt + static_cast<int64_t>(b) * bt_stride + j) : -1;
            if (src < 0 || src >= num_blocks) {
                flag_status(status, PA_DEV_BAD_BLOCK);
                src = min(max(src, 0), num_blocks - 1);
            }
            s_src = src;
        }
        __syncthreads();
        decode_block(kc8, vc8, s_src, pieces_per_block, k, sk, sv);
        __syncthreads();
    }
}

int launch_stage_fp8(const pa_kv_desc *kv, const int32_t *block_tables, int32_t bt_stride,
                     const PlanHeader *hdr, const int *stage_base, const int *stage_list,
                     void *stage_k, void *stage_v, unsigned *status, int grid, cudaStream_t s) {
    if (grid <= 0) return PA_OK;
    // 16 codes per piece; a block holds num_kv_heads * block_size * head_dim codes
    const int pieces = kv->num_kv_heads * kv->block_size * kv->head_dim / 16;
    PdlLaunch l(static_cast<unsigned>(grid), 256, 0, s);
    const cudaError_t e = launch_kernel(
        l, stage_fp8_kernel, static_cast<const uint4 *>(kv->k_cache),
        static_cast<const uint4 *>(kv->v_cache), kv->num_blocks, pieces, block_tables, bt_stride,
        hdr, stage_base, stage_list, static_cast<uint4 *>(stage_k), static_cast<uint4 *>(stage_v),
        status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Cascade decode on an e4m3 pool: the shared prefix's n blocks (list[k],
// k < n) decoded to bf16 staging blocks 0..n-1 for the tensor-core prefix
// pass, which then reads them through the identity list ident[k] = k.
__global__ void __launch_bounds__(256) stage_prefix_fp8_kernel(
    const uint4 *__restrict__ kc8, const uint4 *__restrict__ vc8, int num_blocks,
    int pieces_per_block, const int32_t *__restrict__ list, int n, int32_t *__restrict__ ident,
    uint4 *__restrict__ sk, uint4 *__restrict__ sv, unsigned *status) {
    pdl_wait();  // the list may come from the previous kernel, which may still read the cache
    pdl_trigger();
    for (int k = blockIdx.x; k < n; k += gridDim.x) {
        int64_t src = __ldg(list + k);
        if (src < 0 || src >= num_blocks) {
            if (threadIdx.x == 0) flag_status(status, PA_DEV_BAD_BLOCK);
            src = src < 0 ? 0 : num_blocks - 1;
        }
        if (threadIdx.x == 0) ident[k] = k;
        decode_block(kc8, vc8, src, pieces_per_block, k, sk, sv);
    }
}

int launch_stage_prefix_fp8(const pa_kv_desc *kv, const int32_t *prefix_blocks, int n,
                            int32_t *ident, void *stage_k, void *stage_v, unsigned *status,
                            int grid, cudaStream_t s) {
    if (n <= 0) return PA_OK;
    const int pieces = kv->num_kv_heads * kv->block_size * kv->head_dim / 16;
    PdlLaunch l(static_cast<unsigned>(std::max(1, std::min(grid, n))), 256, 0, s);
    const cudaError_t e = launch_kernel(
        l, stage_prefix_fp8_kernel, static_cast<const uint4 *>(kv->k_cache),
        static_cast<const uint4 *>(kv->v_cache), kv->num_blocks, pieces, prefix_blocks, n, ident,
        static_cast<uint4 *>(stage_k), static_cast<uint4 *>(stage_v), status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
