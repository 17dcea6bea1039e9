// INT8 KV quantiser, shared by the quantising store kernel and the store pass of
// the fused INT8 prefill, so both write the same codes and scales bit for bit.
//
// Source: "面试问答准备: nano-vLLM 推理引擎优化", Q3 (KV cache quantisation):
// each (token, KV head) vector gets scale = max|x| / 127 (floored at 1e-8) and
// codes round(x / scale) in int8; the scale is kept in fp16.  Arithmetic in fp32
// with IEEE division, rounding half away from zero.
//
// Work unit: one warp per (token, group of up to kHeadsPerWarp KV heads).  The
// group's K and V loads are all issued before any arithmetic (more bytes in
// flight per warp than one head's 2 x 2*D), then per head a warp reduction gives
// max|x| and each lane quantises D/32 values of K and of V.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace pa {
namespace quant {

constexpr int kHeadsPerWarp = 4;

// max|x| over the lane's D/32 bf16 values (packed two per word)
template <int D>
__device__ __forceinline__ float lane_absmax(const uint32_t (&r)[D / 64])
{
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e)
        a = fmaxf(a, fabsf(__uint_as_float(e & 1 ? r[e / 2] & 0xffff0000u : r[e / 2] << 16)));
    return a;
}

// Warp-wide max of `a`, the fp32 scale, and the lane's D/32 codes packed in one word.
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

// Quantise token t's K and V rows of heads g0 .. g0 + kHeadsPerWarp - 1 (whole
// warp) into cache row `slot` (0 <= slot < num_blocks * block_size, checked by the
// caller): codes into k_cache/v_cache [slot][Hkv][D], fp16 scales into
// k_scale/v_scale [slot / block_size][Hkv][slot % block_size].
//   k, v: bf16 bits [num_tokens][Hkv][D]
template <int D>
__device__ __forceinline__ void store_token_heads(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                                                  int8_t *__restrict__ k_cache, int8_t *__restrict__ v_cache,
                                                  __half *__restrict__ k_scale, __half *__restrict__ v_scale,
                                                  int32_t t, int g0, int32_t slot, int num_kv_heads, int block_size,
                                                  int lane)
{
    constexpr int E = D / 32; // values per lane
    constexpr int W = E / 2;  // 32-bit words per lane and row
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

} // namespace quant
} // namespace pa
