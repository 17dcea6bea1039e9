// INT8 KV quantiser, shared by the quantising store kernel and the gather of the
// fused INT8 prefill, so both write the same codes and scales bit for bit; and the
// bf16 dequantiser of the INT8 prefill's gather.
//
// Source: "面试问答准备: nano-vLLM 推理引擎优化", Q3 (KV cache quantisation):
// each (token, KV head) vector gets scale = max|x| / 127 (floored at 1e-8) and
// codes round(x / scale) in int8; the scale is kept in fp16.  Arithmetic in fp32
// with IEEE division, rounding half away from zero.
//
// Work unit: kThreadsPerRow<D> adjacent threads per (token, KV head) row (two at
// D = 64, four at D = 128: 32 values per thread): each loads its values (four
// 16-byte loads, all in flight at once), the group combines max|x| with one or
// two shuffles, and each computes the scale and its codes and stores them with
// two 16-byte stores.  A warp quantises 8 or 16 rows side by side, so the
// per-row steps (the max, the scale's division and reciprocal) cost a few
// instructions per row instead of one per lane and row as when a warp shares a
// row, and a thread needs few registers.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace pa {
namespace quant {

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

template <int D>
constexpr int kThreadsPerRow = D / 32;

// The calling thread's 32 values (part h of kThreadsPerRow<D>) of one row of D bf16
// values: four 16-byte loads, issued at once.
struct RowPart {
    uint4 v[4];
};

__device__ __forceinline__ void load_row_part(const uint16_t *__restrict__ row, int h, RowPart &p)
{
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p.v[i] = __ldcs(reinterpret_cast<const uint4 *>(row + 32 * h) + i);
}

// Quantises a loaded part into its 32 codes (c[w] holds codes 4w .. 4w + 3 of the part,
// lowest byte first); returns the row's fp32 scale (the cache keeps its fp16 copy).  The
// kThreadsPerRow<D> threads of a row (adjacent lanes) call it together.
template <int D>
__device__ __forceinline__ float quantise_part(const RowPart &p, uint32_t (&c)[8])
{
    auto word = [&](int e) { // the 32-bit word holding values 2e and 2e + 1
        const uint4 &u = p.v[e >> 2];
        return (e & 3) == 0 ? u.x : (e & 3) == 1 ? u.y : (e & 3) == 2 ? u.z : u.w;
    };
    float m[4]; // a tree of maxima: max is exact, any order gives the same value
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = 0.f;
#pragma unroll
        for (int e = 4 * i; e < 4 * i + 4; ++e) {
            const uint32_t w = word(e);
            m[i] = fmaxf(m[i], fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xffff0000u))));
        }
    }
    float a = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
    // the row's other parts, in the adjacent lanes of the group
    constexpr int TPR = kThreadsPerRow<D>;
    const uint32_t group = ((1u << TPR) - 1) << (threadIdx.x & (32 - TPR));
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1)
        a = fmaxf(a, __shfl_xor_sync(group, a, o));
    const float scale = fmaxf(__fdiv_rn(a, 127.0f), 1e-8f);
    const float rcp = __frcp_rn(scale);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t w0 = word(2 * k), w1 = word(2 * k + 1);
        const int c0 = code_of(__uint_as_float(w0 << 16), scale, rcp);
        const int c1 = code_of(__uint_as_float(w0 & 0xffff0000u), scale, rcp);
        const int c2 = code_of(__uint_as_float(w1 << 16), scale, rcp);
        const int c3 = code_of(__uint_as_float(w1 & 0xffff0000u), scale, rcp);
        c[k] = (uint32_t)(c0 & 0xff) | (uint32_t)(c1 & 0xff) << 8 | (uint32_t)(c2 & 0xff) << 16 |
               (uint32_t)(c3 & 0xff) << 24;
    }
    return scale;
}

// quantise_part, with the 32 codes stored at codes + 32 h (codes: the row's D int8 codes,
// 16-byte aligned).
template <int D>
__device__ __forceinline__ float quantise_row_part(const RowPart &p, int8_t *__restrict__ codes, int h)
{
    uint32_t c[8];
    const float scale = quantise_part<D>(p, c);
    uint4 *dst = reinterpret_cast<uint4 *>(codes + 32 * h);
    dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
    dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    return scale;
}

// Code j of the word (lowest byte first) as an exact fp32 value: the biased code
// (code + 128, the byte xor 0x80) placed in the low mantissa bits of 2^23, minus
// 2^23 + 128.
__device__ __forceinline__ float code_value(uint32_t biased, int j)
{
    return __int_as_float((int)__byte_perm(biased, 0x4B000000u, 0x7540u | (uint32_t)j)) - 8388736.0f;
}

// The 32 codes of a part (as quantise_part returns them) dequantised to bf16:
// RN(code * scale) with the product exact in fp32 (8-bit code, 11-bit fp16 scale),
// i.e. one rounding of the exact value.  out[i] holds values 8i .. 8i + 7, lowest first.
__device__ __forceinline__ void dequantise_part(const uint32_t (&c)[8], float scale, uint4 (&out)[4])
{
    uint32_t v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t b = c[k] ^ 0x80808080u;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const __nv_bfloat162 pair =
                __floats2bfloat162_rn(code_value(b, j) * scale, code_value(b, j + 1) * scale);
            v[2 * k + j / 2] = *reinterpret_cast<const uint32_t *>(&pair);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// Part h (loaded in p) of the K or V row of token t, KV head g, quantised into cache
// row `slot` (0 <= slot < num_blocks * block_size, checked by the caller): codes
// into codes_cache [slot][Hkv][D], the fp16 scale (written by part 0) into scales
// [slot / block_size][Hkv][slot % block_size].
template <int D>
__device__ __forceinline__ void store_row_part(const RowPart &p, int8_t *__restrict__ codes_cache,
                                               __half *__restrict__ scales, int g, int32_t slot, int num_kv_heads,
                                               int block_size, int h)
{
    const float scale = quantise_row_part<D>(p, codes_cache + ((size_t)slot * num_kv_heads + g) * D, h);
    if (h == 0)
        scales[((size_t)(slot / block_size) * num_kv_heads + g) * block_size + slot % block_size] =
            __float2half_rn(scale);
}

} // namespace quant
} // namespace pa
