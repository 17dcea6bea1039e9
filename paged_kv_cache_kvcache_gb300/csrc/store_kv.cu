// KV scatter: copy each new token's K/V rows into its cache slot.
//
// Source: "手搓 vLLM 推理引擎" (LLM-101-CN nano-vllm walkthrough), Step 4,
// "Triton Kernel：写入 KV Cache" — one program per token reads its slot from
// slot_mapping, returns if the slot is -1 (CUDA-graph padding), and copies the
// num_kv_heads*head_dim values of K and of V to cache row `slot`.
//
// GB300 design: one warp per token, 16-byte vector loads/stores, so a warp
// instruction moves 512 contiguous bytes (a 2 KiB Qwen3 row is 4 instructions
// per tensor).  Pure bandwidth work: 2 x (read + write) of the row bytes.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "quant.cuh"

namespace pa {

__device__ uint32_t g_store_error; // 1 = a slot outside [-1, num_slots) was skipped

__global__ void __launch_bounds__(256) store_kvcache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                                            uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                            const int32_t *__restrict__ slot_mapping,
                                                            int32_t num_tokens, int32_t row_vecs, int64_t num_slots)
{
    const int32_t t = (int32_t)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens)
        return;
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0 || slot >= num_slots) {
        if (slot != -1 && lane == 0)
            atomicOr(&g_store_error, 1u);
        return;
    }
    const uint4 *ks = k + (size_t)t * row_vecs;
    const uint4 *vs = v + (size_t)t * row_vecs;
    uint4 *kd = k_cache + (size_t)slot * row_vecs;
    uint4 *vd = v_cache + (size_t)slot * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) {
        uint4 a = __ldcs(ks + i);
        uint4 b = __ldcs(vs + i);
        kd[i] = a;
        vd[i] = b;
    }
}

int launch_store_kvcache(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                         const int32_t *slot_mapping, int32_t num_tokens, void *stream)
{
    const int32_t row_vecs = d.num_kv_heads * d.head_dim * 2 / 16;
    const int threads = 256;
    const int64_t blocks = ((int64_t)num_tokens * 32 + threads - 1) / threads;
    store_kvcache_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), slot_mapping, num_tokens, row_vecs, (int64_t)d.num_blocks * d.block_size);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "store_kvcache launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

// INT8 scatter: the quantiser of quant.cuh, kThreadsPerRow<D> adjacent threads
// per (tensor, token, KV head) row, slots checked as in the bf16 scatter.
template <int D>
__global__ void __launch_bounds__(256) store_kvcache_int8_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, int8_t *__restrict__ k_cache,
    int8_t *__restrict__ v_cache, __half *__restrict__ k_scale, __half *__restrict__ v_scale,
    const int32_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t num_kv_heads, int32_t block_size,
    int64_t num_slots)
{
    constexpr int TPR = quant::kThreadsPerRow<D>;
    const int64_t rows = (int64_t)num_tokens * num_kv_heads; // per tensor
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t i = j / TPR; // the row (both threads of a row leave or stay together)
    if (i >= 2 * rows)
        return;
    const bool is_v = i >= rows;
    const int64_t r = is_v ? i - rows : i;
    const int32_t t = (int32_t)(r / num_kv_heads);
    const int g = (int)(r % num_kv_heads);
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0 || slot >= num_slots) {
        if (slot != -1 && !is_v && g == 0)
            atomicOr(&g_store_error, 1u);
        return;
    }
    const int h = (int)(j % TPR);
    quant::RowPart part;
    quant::load_row_part((is_v ? v : k) + ((size_t)t * num_kv_heads + g) * D, h, part);
    quant::store_row_part<D>(part, is_v ? v_cache : k_cache, is_v ? v_scale : k_scale, g, slot, num_kv_heads,
                             block_size, h);
}

int launch_store_kvcache_int8(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                              void *k_scale, void *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                              void *stream)
{
    const int threads = 256;
    const int64_t blocks = (2 * (int64_t)num_tokens * d.num_kv_heads * (d.head_dim / 32) + threads - 1) / threads;
    auto kern = d.head_dim == 128 ? store_kvcache_int8_kernel<128> : store_kvcache_int8_kernel<64>;
    kern<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
        static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v), static_cast<int8_t *>(k_cache),
        static_cast<int8_t *>(v_cache), static_cast<__half *>(k_scale), static_cast<__half *>(v_scale),
        slot_mapping, num_tokens, d.num_kv_heads, d.block_size, (int64_t)d.num_blocks * d.block_size);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "store_kvcache_int8 launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

int read_store_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_store_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_store_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading store error word: %s", cudaGetErrorString(e));
    *code |= v;
    return PA_OK;
}

} // namespace pa
