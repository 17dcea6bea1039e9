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
// scales are reproducible bit for bit.  One warp per (token, group of up to
// kHeadsPerWarp KV heads): the group's K and V loads are all issued before any
// arithmetic (more bytes in flight per warp than one head's 2 x 2*D), then
// per head a warp reduction gives max|x| and each lane quantises D/32 values
// of K and of V.
constexpr int kHeadsPerWarp = 4;

template <int D>
__device__ __forceinline__ void quantise_lane(const uint32_t (&r)[D / 64], float a, uint32_t &codes, float &scale)
{
    constexpr int E = D / 32; // values per lane
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    scale = fmaxf(__fdiv_rn(a, 127.0f), 1e-8f);
    codes = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float x = __uint_as_float(e & 1 ? r[e / 2] & 0xffff0000u : r[e / 2] << 16);
        const float q = __fdiv_rn(x, scale);
        const int i = __float2int_rz(q >= 0.f ? __fadd_rn(q, 0.5f) : __fsub_rn(q, 0.5f));
        codes |= (uint32_t)(i & 0xff) << (8 * e);
    }
}

template <int D>
__device__ __forceinline__ float lane_absmax(const uint32_t (&r)[D / 64])
{
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e)
        a = fmaxf(a, fabsf(__uint_as_float(e & 1 ? r[e / 2] & 0xffff0000u : r[e / 2] << 16)));
    return a;
}

template <int D>
__global__ void __launch_bounds__(256) store_kvcache_int8_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, int8_t *__restrict__ k_cache,
    int8_t *__restrict__ v_cache, __half *__restrict__ k_scale, __half *__restrict__ v_scale,
    const int32_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t num_kv_heads, int32_t block_size,
    int64_t num_slots)
{
    constexpr int E = D / 32; // values per lane
    constexpr int W = E / 2;  // 32-bit words per lane and row
    const int groups = (num_kv_heads + kHeadsPerWarp - 1) / kHeadsPerWarp;
    const int64_t w = (int64_t)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (int64_t)num_tokens * groups)
        return;
    const int32_t t = (int32_t)(w / groups);
    const int g0 = (int)(w % groups) * kHeadsPerWarp;
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0 || slot >= num_slots) {
        if (slot != -1 && lane == 0 && g0 == 0)
            atomicOr(&g_store_error, 1u);
        return;
    }
    uint32_t rk[kHeadsPerWarp][W], rv[kHeadsPerWarp][W]; // E bf16 values per lane and head
#pragma unroll
    for (int h = 0; h < kHeadsPerWarp; ++h) {
        if (g0 + h >= num_kv_heads)
            break;
        const size_t src = ((size_t)t * num_kv_heads + g0 + h) * D + lane * E;
        if constexpr (E == 4) {
            const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(k + src));
            const uint2 b = __ldcs(reinterpret_cast<const uint2 *>(v + src));
            rk[h][0] = a.x, rk[h][1] = a.y, rv[h][0] = b.x, rv[h][1] = b.y;
        } else {
            rk[h][0] = __ldcs(reinterpret_cast<const unsigned int *>(k + src));
            rv[h][0] = __ldcs(reinterpret_cast<const unsigned int *>(v + src));
        }
    }
#pragma unroll
    for (int h = 0; h < kHeadsPerWarp; ++h) {
        const int g = g0 + h;
        if (g >= num_kv_heads)
            break;
        uint32_t ck, cv;
        float sk, sv;
        quantise_lane<D>(rk[h], lane_absmax<D>(rk[h]), ck, sk);
        quantise_lane<D>(rv[h], lane_absmax<D>(rv[h]), cv, sv);
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
}

int launch_store_kvcache_int8(const pa_dims &d, const void *k, const void *v, void *k_cache, void *v_cache,
                              void *k_scale, void *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                              void *stream)
{
    const int threads = 256;
    const int64_t groups = (d.num_kv_heads + kHeadsPerWarp - 1) / kHeadsPerWarp;
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
