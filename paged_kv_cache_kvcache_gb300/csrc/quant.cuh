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

// code = trunc(q + 0.5 * sign(q)) with q = x / scale rounded to nearest (IEEE
// division).  The division is only carried out where it can matter: q' = x *
// RN(1 / scale) differs from q by at most about 3 ulp(q) (two roundings of
// relative size 2^-24 against q's one), and the code only changes where q
// crosses a half-integer, so when q' lies more than |q'| * 2^-20 (>= 8 ulp) from
// every half-integer, q' gives the same code as q.  Otherwise (rare; always for
// exact half-integers) q itself is computed.  NaN and infinite quotients take
// the same value on both routes.
__device__ __forceinline__ int code_of(float x, float scale, float rcp)
{
    float q = __fmul_rn(x, rcp);
    const float aq = fabsf(q);
    // distance of |q'| to the nearest half-integer (exact: Sterbenz, or far from 0.5)
    const float d = fabsf(__fsub_rn(__fsub_rn(aq, floorf(aq)), 0.5f));
    if (d < aq * 0x1p-20f)
        q = __fdiv_rn(x, scale);
    return __float2int_rz(q >= 0.f ? __fadd_rn(q, 0.5f) : __fsub_rn(q, 0.5f));
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
    const float rcp = __frcp_rn(scale);
    codes = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float x = __uint_as_float(e & 1 ? r[e / 2] & 0xffff0000u : r[e / 2] << 16);
        codes |= (uint32_t)(code_of(x, scale, rcp) & 0xff) << (8 * e);
    }
}

// Token t's K and V rows of heads g0 .. g0 + kHeadsPerWarp - 1 into registers
// (whole warp; D/32 bf16 values per lane and head).  k, v: bf16 bits [tokens][Hkv][D].
template <int D>
struct HeadRows {
    uint32_t k[kHeadsPerWarp][D / 64], v[kHeadsPerWarp][D / 64];
};

template <int D>
__device__ __forceinline__ void load_token_heads(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                                                 int32_t t, int g0, int num_kv_heads, int lane, HeadRows<D> &r)
{
    constexpr int E = D / 32; // values per lane
#pragma unroll
    for (int h = 0; h < kHeadsPerWarp; ++h) {
        if (g0 + h >= num_kv_heads)
            break;
        const size_t src = ((size_t)t * num_kv_heads + g0 + h) * D + lane * E;
        if constexpr (E == 4) {
            const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(k + src));
            const uint2 b = __ldcs(reinterpret_cast<const uint2 *>(v + src));
            r.k[h][0] = a.x, r.k[h][1] = a.y, r.v[h][0] = b.x, r.v[h][1] = b.y;
        } else {
            r.k[h][0] = __ldcs(reinterpret_cast<const unsigned int *>(k + src));
            r.v[h][0] = __ldcs(reinterpret_cast<const unsigned int *>(v + src));
        }
    }
}

// Quantise loaded rows into cache row `slot` (0 <= slot < num_blocks * block_size,
// checked by the caller): codes into k_cache/v_cache [slot][Hkv][D], fp16 scales
// into k_scale/v_scale [slot / block_size][Hkv][slot % block_size].
template <int D>
__device__ __forceinline__ void quantise_token_heads(const HeadRows<D> &r, int8_t *__restrict__ k_cache,
                                                     int8_t *__restrict__ v_cache, __half *__restrict__ k_scale,
                                                     __half *__restrict__ v_scale, int g0, int32_t slot,
                                                     int num_kv_heads, int block_size, int lane)
{
    constexpr int E = D / 32; // values per lane
#pragma unroll
    for (int h = 0; h < kHeadsPerWarp; ++h) {
        const int g = g0 + h;
        if (g >= num_kv_heads)
            break;
        uint32_t ck, cv;
        float sk, sv;
        quantise_lane<D>(r.k[h], lane_absmax<D>(r.k[h]), ck, sk);
        quantise_lane<D>(r.v[h], lane_absmax<D>(r.v[h]), cv, sv);
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
