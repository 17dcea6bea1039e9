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

// INT8 scatter: the quantiser of quant.cuh (one warp per token and group of up
// to quant::kHeadsPerWarp KV heads), slots checked as in the bf16 scatter.
template <int D>
__global__ void __launch_bounds__(256) store_kvcache_int8_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, int8_t *__restrict__ k_cache,
    int8_t *__restrict__ v_cache, __half *__restrict__ k_scale, __half *__restrict__ v_scale,
    const int32_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t num_kv_heads, int32_t block_size,
    int64_t num_slots)
{
    const int groups = (num_kv_heads + quant::kHeadsPerWarp - 1) / quant::kHeadsPerWarp;
    const int64_t w = (int64_t)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (int64_t)num_tokens * groups)
        return;
    const int32_t t = (int32_t)(w / groups);
    const int g0 = (int)(w % groups) * quant::kHeadsPerWarp;
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0 || slot >= num_slots) {
        if (slot != -1 && lane == 0 && g0 == 0)
            atomicOr(&g_store_error, 1u);
        return;
    }
    quant::HeadRows<D> r;
    quant::load_token_heads<D>(k, v, t, g0, num_kv_heads, lane, r);
    quant::quantise_token_heads<D>(r, k_cache, v_cache, k_scale, v_scale, g0, slot, num_kv_heads, block_size, lane);
}

int launch_store_kvcache_int8(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                              void *k_scale, void *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                              void *stream)
{
    const int threads = 256;
    const int64_t groups = (d.num_kv_heads + quant::kHeadsPerWarp - 1) / quant::kHeadsPerWarp;
    const int64_t blocks = ((int64_t)num_tokens * groups * 32 + threads - 1) / threads;
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
