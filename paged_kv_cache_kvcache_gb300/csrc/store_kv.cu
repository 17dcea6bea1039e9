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

// INT8 scatter.  Source: "面试问答准备: nano-vLLM 推理引擎优化", Q3 (KV cache
// quantisation): each head vector gets scale = max|x| / 127 (floored at 1e-8)
// and codes round(x / scale) in int8; the scale is kept in fp16.  Arithmetic
// in fp32 with IEEE division, rounding half away from zero, so codes and
// scales are reproducible bit for bit.  One warp per (token, KV head): a warp
// reduction gives max|x|; each lane quantises D/32 values of K and of V.
template <int D>
__global__ void __launch_bounds__(256) store_kvcache_int8_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, int8_t *__restrict__ k_cache,
    int8_t *__restrict__ v_cache, __half *__restrict__ k_scale, __half *__restrict__ v_scale,
    const int32_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t num_kv_heads, int32_t block_size,
    int64_t num_slots)
{
    constexpr int E = D / 32; // values per lane
    const int64_t w = (int64_t)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (int64_t)num_tokens * num_kv_heads)
        return;
    const int32_t t = (int32_t)(w / num_kv_heads);
    const int g = (int)(w % num_kv_heads);
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0 || slot >= num_slots) {
        if (slot != -1 && lane == 0 && g == 0)
            atomicOr(&g_store_error, 1u);
        return;
    }
    const size_t src = ((size_t)t * num_kv_heads + g) * D + lane * E;
    uint32_t rk[E / 2], rv[E / 2]; // E bf16 values per lane, one 4- or 8-byte load
    if constexpr (E == 4) {
        const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(k + src));
        const uint2 b = __ldcs(reinterpret_cast<const uint2 *>(v + src));
        rk[0] = a.x, rk[1] = a.y, rv[0] = b.x, rv[1] = b.y;
    } else {
        rk[0] = __ldcs(reinterpret_cast<const unsigned int *>(k + src));
        rv[0] = __ldcs(reinterpret_cast<const unsigned int *>(v + src));
    }
    float xk[E], xv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        xk[e] = __uint_as_float(e & 1 ? rk[e / 2] & 0xffff0000u : rk[e / 2] << 16);
        xv[e] = __uint_as_float(e & 1 ? rv[e / 2] & 0xffff0000u : rv[e / 2] << 16);
    }
    float ak = 0.f, av = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        ak = fmaxf(ak, fabsf(xk[e]));
        av = fmaxf(av, fabsf(xv[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, o));
        av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
    }
    const float sk = fmaxf(__fdiv_rn(ak, 127.0f), 1e-8f);
    const float sv = fmaxf(__fdiv_rn(av, 127.0f), 1e-8f);
    uint32_t ck = 0, cv = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float qk = __fdiv_rn(xk[e], sk), qv = __fdiv_rn(xv[e], sv);
        const int ik = __float2int_rz(qk >= 0.f ? __fadd_rn(qk, 0.5f) : __fsub_rn(qk, 0.5f));
        const int iv = __float2int_rz(qv >= 0.f ? __fadd_rn(qv, 0.5f) : __fsub_rn(qv, 0.5f));
        ck |= (uint32_t)(ik & 0xff) << (8 * e);
        cv |= (uint32_t)(iv & 0xff) << (8 * e);
    }
    const size_t dst = ((size_t)slot * num_kv_heads + g) * D + lane * E;
    if constexpr (E == 4) {
        *reinterpret_cast<uint32_t *>(k_cache + dst) = ck;
        *reinterpret_cast<uint32_t *>(v_cache + dst) = cv;
    } else {
        *reinterpret_cast<uint16_t *>(k_cache + dst) = (uint16_t)ck;
        *reinterpret_cast<uint16_t *>(v_cache + dst) = (uint16_t)cv;
    }
    if (lane == 0) {
        const size_t si = ((size_t)(slot / block_size) * num_kv_heads + g) * block_size + slot % block_size;
        k_scale[si] = __float2half_rn(sk);
        v_scale[si] = __float2half_rn(sv);
    }
}

int launch_store_kvcache_int8(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                              void *k_scale, void *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                              void *stream)
{
    const int threads = 256;
    const int64_t blocks = ((int64_t)num_tokens * d.num_kv_heads * 32 + threads - 1) / threads;
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
