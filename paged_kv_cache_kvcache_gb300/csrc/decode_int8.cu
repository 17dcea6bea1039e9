// Batched single-token GQA decode over an INT8 paged KV cache, dequantisation
// fused into the attention loads; split-KV + LSE combine as in the bf16 decode.
//
// Sources (page title, section):
//  - "面试问答准备: nano-vLLM 推理引擎优化", Q3 (KV cache quantisation): K and
//    V are kept as int8 codes with one scale per token and KV head; the
//    attention kernel dequantises as it reads, so decode moves half the bytes
//    of the bf16 cache.  The cached value is code * scale.
//  - the same page's Q3 follow-ups (Split-K with a log-sum-exp merge), and
//    "推理系统", "瓶颈不是算力，是带宽" (decode time = bytes read / bandwidth).
//
// GB300 design.  Work items, CTA/warp decomposition, cp.async pipeline,
// online softmax, warp merge and partial format are those of the bf16 decode;
// what changes is the operand path:
//  * Each warp owns a ring of stages fed by TMA: for every 16-token chunk its
//    lane 0 issues one 3-D tensor copy of the K codes (16 token rows of D bytes
//    for one KV head, hardware-swizzled), one of the V codes and two 32-byte
//    bulk copies of the chunk's fp16 K and V scales, all completing on the
//    stage's mbarrier (waits are bounded).  A chunk never crosses a block, so a
//    tail chunk's extra rows are in-bounds cache memory; their scores are
//    masked and their V scales zeroed before use.
//  * A code x converts to fp16 exactly: the bit pattern 0x6400 | (x + 128) is
//    1024 + x + 128, minus 1152 gives x (one prmt + one f16x2 subtract per
//    pair).  Both MMAs therefore run as f16 m16n8k16 with fp32 accumulation:
//        S^T[16 tok x 8 heads] = K_codes . Q^T,  then s *= k_scale[tok]
//        O^T[D x 8 heads]     += V_codes^T . (P * v_scale[tok])^T
//    The softmax normaliser sums the unscaled P.  P * v_scale never exceeds
//    the fp16 scale itself (P <= 1), so it stays in fp16 range.
//  * Q is rounded to fp16 once per CTA (exact for bf16 values of magnitude in
//    [2^-14, 65504], clamped beyond).
//  * Operand order: the MMA contraction and the O^T rows may be permuted at
//    will (undone when O is written), so each lane's K codes for all k-steps
//    are one contiguous run of its token row (two 16-byte loads), and its V
//    codes for all d-tiles are one contiguous run of each of its four token
//    rows.  Byte interleaving for V's token pairs is one prmt per word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecLayout8 {
    static constexpr int kChunkBytes = 16 * D;          // 16 tokens of int8 codes
    static constexpr int kStageBytes = 2 * kChunkBytes; // K codes, V codes
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kScaleOff = kWarps * kWarpBytes; // [warp][stage]: 16 K + 16 V fp16 scales
    static constexpr int kBarOff = kScaleOff + kWarps * kStages * 64;
    static constexpr int kUsed = kBarOff + kWarps * kStages * 8;
    static constexpr int kSmemBytes = kUsed + 1024; // + slack to align the base to the swizzle atom
    static constexpr uint32_t kTxBytes = 2 * kChunkBytes + 64;
};

// Byte offset of 16-byte vector v of token t inside a staged chunk, as the TMA
// swizzle writes it: 128-byte rows (D = 128) under SWIZZLE_128B, 64-byte rows
// (D = 64) under SWIZZLE_64B.  The fragment loads below are conflict-free at
// D = 128 (two-way on V at D = 64).
template <int D>
__device__ __forceinline__ uint32_t swz(int t, int v)
{
    if constexpr (D == 128)
        return (uint32_t)(t * 128 + ((v ^ (t & 7)) << 4));
    else
        return (uint32_t)(t * 64 + ((v ^ ((t >> 1) & 3)) << 4));
}

__device__ uint32_t g_decode_error; // bit 0: a bounded wait timed out

constexpr uint32_t kFlip = 0x80808080u;  // int8 -> offset binary (x + 128), per byte
constexpr uint32_t kLoPair = 0x4140u;    // prmt: bytes 0, 1 under 0x64 high bytes
constexpr uint32_t kHiPair = 0x4342u;    // prmt: bytes 2, 3 under 0x64 high bytes
constexpr uint32_t kMagic = 0x64806480u; // f16x2 (1152, 1152)

// Two offset-binary codes of u (chosen by sel) -> f16x2 of the signed codes, exact.
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t u, uint32_t sel)
{
    return ptx::sub_f16x2(ptx::prmt(u, 0x64646464u, sel), kMagic);
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    const float lo = fminf(fmaxf(__uint_as_float(w << 16), -65504.f), 65504.f);
    const float hi = fminf(fmaxf(__uint_as_float(w & 0xffff0000u), -65504.f), 65504.f);
    return ptx::pack_f16(lo, hi);
}

__device__ __forceinline__ float lds_half(uint32_t addr) { return __half2float(__ushort_as_half(ptx::lds_u16(addr))); }

struct DecParams8 {
    const __nv_bfloat16 *q;
    const __half *k_scale;
    const __half *v_scale;
    const int32_t *block_tables;
    const int4 *items;
    __nv_bfloat16 *out;
    float *part_o;
    float *part_lse;
    float scale_log2;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t block_size;
    int32_t max_blocks;
    // fused store (FUSED kernels only): the new token's bf16 K/V rows, where they go, the context lengths
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    int8_t *k_codes_out;
    int8_t *v_codes_out;
    __half *k_scale_out;
    __half *v_scale_out;
    const int32_t *slot_mapping;
    const int32_t *context_lens;
    int64_t num_slots;
};

__device__ uint32_t g_fused8_error; // bit 0: a fused-store slot outside [-1, num_slots) was skipped

// The INT8 quantiser of pa_store_kvcache_int8 on one (token, KV head) row held
// by a warp (D/32 values per lane): returns the codes packed in one word and
// the fp32 scale; the same scale and the same per-value code (quant::code_of)
// as the store kernel, bit for bit.
template <int D>
__device__ __forceinline__ uint32_t quantise_row(const float (&x)[D / 32], float &scale)
{
    constexpr int E = D / 32;
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
        a = fmaxf(a, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    scale = fmaxf(__fdiv_rn(a, 127.0f), 1e-8f);
    const float rcp = __frcp_rn(scale);
    uint32_t codes = 0;
#pragma unroll
    for (int e = 0; e < E; ++e)
        codes |= (uint32_t)(quant::code_of(x[e], scale, rcp) & 0xff) << (8 * e);
    return codes;
}

// FUSED: the CTA whose work item ends at the sequence's last key (the token
// being decoded) quantises that token's K/V rows of its head, writes codes and
// scales into the cache slot and takes the key from its own registers (the
// dequantised values the cache now holds) instead of from the cache.
template <int D, int NT, bool FUSED>
__global__ void __launch_bounds__(kWarps * 32, NT == 1 ? 4 : 3)
    decode_int8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecParams8 p)
{
    using L = DecLayout8<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw); // generic pointer to the aligned base
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int4 item = p.items[blockIdx.x / p.num_kv_heads];
    const int b = item.x, k0 = item.y, pslot = item.w;
    // FUSED: does this item hold the new token?  Then the cache supplies keys k0 .. ctx-2.
    const bool has_new = FUSED && item.z > 0 && item.z == __ldg(p.context_lens + b);
    const int k1 = has_new ? item.z - 1 : item.z;
    const int g = blockIdx.x % p.num_kv_heads;
    const int G = p.group;
    const int Hq = p.num_heads;

    const int nchunks = (k1 - k0 + 15) >> 4;
    const int my_n = nchunks > warp ? (nchunks - warp + kWarps - 1) / kWarps : 0;
    const uint32_t wbase = sbase + warp * L::kWarpBytes;
    const uint32_t sc_base = sbase + L::kScaleOff + warp * kStages * 64;
    const uint32_t bar_base = sbase + L::kBarOff + warp * kStages * 8;
    const int32_t *bt_row = p.block_tables + (size_t)b * p.max_blocks;
    const int bs = p.block_size;
    const int Hkv = p.num_kv_heads;
    int blk_cache = 0;

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s)
            ptx::mbar_init(bar_base + 8 * s, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    __syncwarp();

    // Chunk i of this warp into stage i % kStages (whole warp: the block id comes by shuffle).
    auto issue = [&](int i) {
        if ((i & 31) == 0) { // refresh the block ids of local chunks i .. i+31, one per lane
            const int key = k0 + 16 * (warp + kWarps * (i + lane));
            blk_cache = key < k1 ? __ldg(bt_row + key / bs) : 0;
        }
        const int phys = __shfl_sync(0xffffffffu, blk_cache, i & 31);
        if (lane == 0) {
            const int key0 = k0 + 16 * (warp + kWarps * i);
            const int off0 = key0 & (bs - 1); // a chunk never crosses a block (bs >= 16, key0 % 16 == 0)
            const int st = i % kStages;
            const uint32_t bar = bar_base + 8 * st;
            const uint32_t dst = wbase + st * L::kStageBytes;
            const size_t si = ((size_t)phys * Hkv + g) * bs + off0;
            ptx::mbar_arrive_expect_tx(bar, L::kTxBytes);
            ptx::tma_load_3d(dst, &tm_k, bar, 0, g, phys * bs + off0);
            ptx::tma_load_3d(dst + L::kChunkBytes, &tm_v, bar, 0, g, phys * bs + off0);
            ptx::bulk_load(sc_base + st * 64, p.k_scale + si, 32u, bar);
            ptx::bulk_load(sc_base + st * 64 + 32, p.v_scale + si, 32u, bar);
        }
    };

    // first stages in flight before Q is fetched, so the two latencies overlap
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s)
        if (s < my_n)
            issue(s);

    // Q^T fragments (f16), B operand of the score MMA.  k-step kk of lane c
    // covers d = c*D/4 + 4kk + {0,1} (logical k 2c, 2c+1) and + {2,3} (2c+8, 2c+9).
    uint32_t qf[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hl = nt * 8 + r;
        const bool valid = hl < G;
        const uint2 *qrow = reinterpret_cast<const uint2 *>(
            p.q + ((size_t)b * Hq + (size_t)g * G + (valid ? hl : 0)) * D + c * (D / 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint2 w = valid ? __ldg(qrow + kk) : make_uint2(0u, 0u);
            qf[nt][kk][0] = bf16x2_to_f16x2(w.x);
            qf[nt][kk][1] = bf16x2_to_f16x2(w.y);
        }
    }

    float acc[NT][D / 16][4];
    float m_r[NT][2], l_r[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_r[nt][0] = m_r[nt][1] = -INFINITY;
        l_r[nt][0] = l_r[nt][1] = 0.f;
#pragma unroll
        for (int mi = 0; mi < D / 16; ++mi)
            acc[nt][mi][0] = acc[nt][mi][1] = acc[nt][mi][2] = acc[nt][mi][3] = 0.f;
    }


    int done = 0; // chunks consumed (all issued chunks are waited for before exit)
    for (int i = 0; i < my_n; ++i) {
        // stage (i - 1) % kStages was read by every lane in the previous iteration
        __syncwarp();
        if (i + kStages - 1 < my_n)
            issue(i + kStages - 1);
        const int st = i % kStages;
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_base + 8 * st, (uint32_t)(i / kStages) & 1u))) {
            if (lane == 0)
                atomicOr(&g_decode_error, 1u);
            break;
        }
        done = i + 1;

        const uint32_t kb = wbase + st * L::kStageBytes;
        const uint32_t vb = kb + L::kChunkBytes;
        const uint32_t sb = sc_base + st * 64;
        const int key0 = k0 + 16 * (warp + kWarps * i);

        // K codes of tokens r and r + 8: bytes [c*D/4, (c+1)*D/4) of each row
        uint32_t kw[2][D / 16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = r + 8 * h;
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
                const uint4 u = ptx::lds_v4(kb + swz<D>(t, (D / 64) * c + x));
                kw[h][4 * x] = u.x, kw[h][4 * x + 1] = u.y, kw[h][4 * x + 2] = u.z, kw[h][4 * x + 3] = u.w;
            }
        }
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t u0 = kw[0][kk] ^ kFlip, u1 = kw[1][kk] ^ kFlip;
            const uint32_t a0 = codes_to_f16x2(u0, kLoPair), a2 = codes_to_f16x2(u0, kHiPair);
            const uint32_t a1 = codes_to_f16x2(u1, kLoPair), a3 = codes_to_f16x2(u1, kHiPair);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                ptx::mma_16816_f16(sc[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
        }

        const float ks0 = lds_half(sb + 2 * r) * p.scale_log2;
        const float ks1 = lds_half(sb + 2 * (r + 8)) * p.scale_log2;
        const bool v0 = key0 + r < k1;
        const bool v1 = key0 + r + 8 < k1;
        const float vs0 = v0 ? lds_half(sb + 32 + 2 * r) : 0.f; // rows past the context: weight 0
        const float vs1 = v1 ? lds_half(sb + 32 + 2 * (r + 8)) : 0.f;
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float s0 = v0 ? sc[nt][0] * ks0 : -INFINITY;
            const float s1 = v0 ? sc[nt][1] * ks0 : -INFINITY;
            const float s2 = v1 ? sc[nt][2] * ks1 : -INFINITY;
            const float s3 = v1 ? sc[nt][3] * ks1 : -INFINITY;
            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m_r[nt][0], mx0), mn1 = fmaxf(m_r[nt][1], mx1);
            const float al0 = ptx::ex2(m_r[nt][0] - mn0), al1 = ptx::ex2(m_r[nt][1] - mn1);
            m_r[nt][0] = mn0;
            m_r[nt][1] = mn1;
            const float p0 = ptx::ex2(s0 - mn0), p1 = ptx::ex2(s1 - mn1);
            const float p2 = ptx::ex2(s2 - mn0), p3 = ptx::ex2(s3 - mn1);
            l_r[nt][0] = l_r[nt][0] * al0 + p0 + p2;
            l_r[nt][1] = l_r[nt][1] * al1 + p1 + p3;
            if (__any_sync(0xffffffffu, (al0 != 1.f) | (al1 != 1.f))) { // skipped while no row max moves
#pragma unroll
                for (int mi = 0; mi < D / 16; ++mi) {
                    acc[nt][mi][0] *= al0;
                    acc[nt][mi][1] *= al1;
                    acc[nt][mi][2] *= al0;
                    acc[nt][mi][3] *= al1;
                }
            }
            pb[nt][0] = ptx::movmatrix_trans(ptx::pack_f16(p0 * vs0, p1 * vs0));
            pb[nt][1] = ptx::movmatrix_trans(ptx::pack_f16(p2 * vs1, p3 * vs1));
        }

        // V codes of tokens 2c, 2c+1, 2c+8, 2c+9: bytes [r*D/8, (r+1)*D/8) of each
        // row.  Byte 2*mi + hi of that run is d-row (mi, r + 8*hi) of O^T tile mi.
        uint32_t vw[4][D / 32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = 2 * c + (j & 1) + 8 * (j >> 1);
            if constexpr (D == 128) {
                const uint4 u = ptx::lds_v4(vb + swz<D>(t, r));
                vw[j][0] = u.x, vw[j][1] = u.y, vw[j][2] = u.z, vw[j][3] = u.w;
            } else {
                const uint2 u = ptx::lds_v2(vb + swz<D>(t, r >> 1) + (r & 1) * 8);
                vw[j][0] = u.x, vw[j][1] = u.y;
            }
        }
#pragma unroll
        for (int w = 0; w < D / 32; ++w) {
            // token pairs (2c, 2c+1) and (2c+8, 2c+9) interleaved byte by byte
            const uint32_t x01 = ptx::prmt(vw[0][w], vw[1][w], 0x5140u) ^ kFlip; // tile 2w
            const uint32_t y01 = ptx::prmt(vw[0][w], vw[1][w], 0x7362u) ^ kFlip; // tile 2w + 1
            const uint32_t x89 = ptx::prmt(vw[2][w], vw[3][w], 0x5140u) ^ kFlip;
            const uint32_t y89 = ptx::prmt(vw[2][w], vw[3][w], 0x7362u) ^ kFlip;
            {
                const uint32_t a0 = codes_to_f16x2(x01, kLoPair), a1 = codes_to_f16x2(x01, kHiPair);
                const uint32_t a2 = codes_to_f16x2(x89, kLoPair), a3 = codes_to_f16x2(x89, kHiPair);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    ptx::mma_16816_f16(acc[nt][2 * w], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
            {
                const uint32_t a0 = codes_to_f16x2(y01, kLoPair), a1 = codes_to_f16x2(y01, kHiPair);
                const uint32_t a2 = codes_to_f16x2(y89, kLoPair), a3 = codes_to_f16x2(y89, kHiPair);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    ptx::mma_16816_f16(acc[nt][2 * w + 1], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
        }
    }
    // after a timed-out wait: let the copies still in flight land (bounded) before the buffers are reused
    for (int i = done; i < my_n && i < done + kStages; ++i)
        ptx::mbar_wait(bar_base + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u);

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int o = 4; o < 32; o <<= 1)
                l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], o);

    // merge the 4 warps through shared memory (pipeline buffers are free now)
    __syncthreads();
    constexpr int H8 = 8 * NT;
    constexpr int kRow = D + 4; // padded head row (floats): the float4 stores below conflict at most 2-way
    float *mrg_m = reinterpret_cast<float *>(smem);
    float *mrg_l = mrg_m + kWarps * H8;
    float *mrg_o = mrg_l + kWarps * H8; // [warp][head][kRow], d in natural order
    float *s_new = mrg_o + (size_t)kWarps * H8 * kRow; // FUSED: the new key's score per head (log2 units)
    float *v_new = s_new + H8;                         // FUSED: the new value, dequantised
    if constexpr (FUSED) {
        if (has_new && warp < 2) {
            // warp 0 quantises K, warp 1 V: codes and fp16 scale into the slot, dequantised values kept
            constexpr int E = D / 32;
            const size_t row = ((size_t)b * p.num_kv_heads + g) * D + lane * E;
            const __nv_bfloat16 *src = (warp == 0 ? p.k_new : p.v_new) + row;
            float x[E];
#pragma unroll
            for (int e = 0; e < E; ++e)
                x[e] = __bfloat162float(src[e]);
            float sc;
            const uint32_t codes = quantise_row<D>(x, sc);
            const __half sc16 = __float2half_rn(sc);
            const float deq = __half2float(sc16);
            float xd[E];
#pragma unroll
            for (int e = 0; e < E; ++e)
                xd[e] = (float)(int8_t)(codes >> (8 * e)) * deq;
            const int32_t slot = __ldg(p.slot_mapping + b);
            if (slot >= 0 && slot < p.num_slots) {
                const size_t dst = ((size_t)slot * p.num_kv_heads + g) * D + lane * E;
                int8_t *cd = (warp == 0 ? p.k_codes_out : p.v_codes_out) + dst;
                if constexpr (E == 4)
                    *reinterpret_cast<uint32_t *>(cd) = codes;
                else
                    *reinterpret_cast<uint16_t *>(cd) = (uint16_t)codes;
                if (lane == 0) {
                    const int bs = p.block_size;
                    (warp == 0 ? p.k_scale_out : p.v_scale_out)[((size_t)(slot / bs) * p.num_kv_heads + g) * bs +
                                                                slot % bs] = sc16;
                }
            } else if (slot != -1 && lane == 0) {
                atomicOr(&g_fused8_error, 1u);
            }
            if (warp == 0) { // the new key's score for every head of the group
                for (int hl = 0; hl < G; ++hl) {
                    const __nv_bfloat16 *qr = p.q + ((size_t)b * Hq + (size_t)g * G + hl) * D + lane * E;
                    float acc_s = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        acc_s += __bfloat162float(qr[e]) * xd[e];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        acc_s += __shfl_xor_sync(0xffffffffu, acc_s, o);
                    if (lane == 0)
                        s_new[hl] = acc_s * p.scale_log2;
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    v_new[lane * E + e] = xd[e];
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int h0 = nt * 8 + 2 * c;
        if (lane < 4) {
            mrg_m[warp * H8 + h0] = m_r[nt][0];
            mrg_m[warp * H8 + h0 + 1] = m_r[nt][1];
            mrg_l[warp * H8 + h0] = l_r[nt][0];
            mrg_l[warp * H8 + h0 + 1] = l_r[nt][1];
        }
        // O^T row (mi, r + 8*hi) is d = r*D/8 + 2*mi + hi: this lane's D/8 values per head are contiguous
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float4 *dst = reinterpret_cast<float4 *>(mrg_o + ((size_t)warp * H8 + h0 + j) * kRow + r * (D / 8));
#pragma unroll
            for (int v = 0; v < D / 32; ++v)
                dst[v] = make_float4(acc[nt][2 * v][j], acc[nt][2 * v][j + 2], acc[nt][2 * v + 1][j],
                                     acc[nt][2 * v + 1][j + 2]);
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int hl = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            M = fmaxf(M, mrg_m[w * H8 + hl]);
        float Lsum = 0.f, O = 0.f;
        if (FUSED && has_new)
            M = fmaxf(M, s_new[hl]);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = ptx::ex2(mrg_m[w * H8 + hl] - M);
                Lsum += f * mrg_l[w * H8 + hl];
                O += f * mrg_o[((size_t)w * H8 + hl) * kRow + d];
            }
            if (FUSED && has_new) { // the new token: weight 2^(s - M), its dequantised value
                const float f = ptx::ex2(s_new[hl] - M);
                Lsum += f;
                O += f * v_new[d];
            }
        }
        const float o = Lsum > 0.f ? O / Lsum : 0.f;
        const size_t h = (size_t)g * G + hl;
        if (pslot < 0) {
            p.out[((size_t)b * Hq + h) * D + d] = __float2bfloat16_rn(o);
        } else {
            p.part_o[((size_t)pslot * Hq + h) * D + d] = o;
            if (d == 0)
                p.part_lse[(size_t)pslot * Hq + h] = Lsum > 0.f ? M + __log2f(Lsum) : -INFINITY;
        }
    }
}

template <int D, int NT, bool FUSED>
int launch_int8(const DecodeArgs &a, const DecParams8 &p, cudaStream_t stream)
{
    if (int rc = ensure_smem<decode_int8_kernel<D, NT, FUSED>>(DecLayout8<D>::kSmemBytes, "decode_int8"))
        return rc;
    // codes as uint8 [num_slots][Hkv][D]: box = one head's D bytes x 16 token rows
    const pa_dims &d = a.dims;
    const uint64_t rows = (uint64_t)d.num_blocks * d.block_size;
    const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap tk, tv;
    int rc;
    if ((rc = encode_tmap_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_cache, D, d.num_kv_heads, rows, D,
                             (uint64_t)d.num_kv_heads * D, D, 1, 16, sw, "int8 k_cache")) != PA_OK)
        return rc;
    if ((rc = encode_tmap_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v_cache, D, d.num_kv_heads, rows, D,
                             (uint64_t)d.num_kv_heads * D, D, 1, 16, sw, "int8 v_cache")) != PA_OK)
        return rc;
    // flat grid, heads of one work item adjacent: they read neighbouring
    // segments of the same token rows at about the same time (DRAM locality)
    dim3 grid((unsigned)(a.num_items * a.dims.num_kv_heads));
    decode_int8_kernel<D, NT, FUSED><<<grid, kWarps * 32, DecLayout8<D>::kSmemBytes, stream>>>(tk, tv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "decode_int8 launch: %s", cudaGetErrorString(e));
    return launch_decode_combine(a, stream);
}

} // namespace

int launch_decode_int8(const DecodeArgs &a, void *stream)
{
    DecParams8 p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k_scale = static_cast<const __half *>(a.k_scale);
    p.v_scale = static_cast<const __half *>(a.v_scale);
    p.block_tables = a.block_tables;
    p.items = reinterpret_cast<const int4 *>(a.items);
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.part_o = a.part_o;
    p.part_lse = a.part_lse;
    p.scale_log2 = a.scale * kLog2e;
    p.num_heads = a.dims.num_heads;
    p.num_kv_heads = a.dims.num_kv_heads;
    p.group = a.dims.num_heads / a.dims.num_kv_heads;
    p.block_size = a.dims.block_size;
    p.max_blocks = a.max_blocks_per_seq;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool two = p.group > 8;
    if (a.k_new) { // fused quantising store + decode
        p.k_new = static_cast<const __nv_bfloat16 *>(a.k_new);
        p.v_new = static_cast<const __nv_bfloat16 *>(a.v_new);
        p.k_codes_out = static_cast<int8_t *>(const_cast<void *>(a.k_cache));
        p.v_codes_out = static_cast<int8_t *>(const_cast<void *>(a.v_cache));
        p.k_scale_out = static_cast<__half *>(const_cast<void *>(a.k_scale));
        p.v_scale_out = static_cast<__half *>(const_cast<void *>(a.v_scale));
        p.slot_mapping = a.slot_mapping;
        p.context_lens = a.context_lens;
        p.num_slots = (int64_t)a.dims.num_blocks * a.dims.block_size;
        if (a.dims.head_dim == 128)
            return two ? launch_int8<128, 2, true>(a, p, s) : launch_int8<128, 1, true>(a, p, s);
        return two ? launch_int8<64, 2, true>(a, p, s) : launch_int8<64, 1, true>(a, p, s);
    }
    if (a.dims.head_dim == 128)
        return two ? launch_int8<128, 2, false>(a, p, s) : launch_int8<128, 1, false>(a, p, s);
    return two ? launch_int8<64, 2, false>(a, p, s) : launch_int8<64, 1, false>(a, p, s);
}

int read_fused8_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fused8_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_fused8_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading fused-store error word: %s", cudaGetErrorString(e));
    *code |= v; // same meaning as the store kernels' bit 0
    return PA_OK;
}

int read_decode_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_decode_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading decode error word: %s", cudaGetErrorString(e));
    *code |= v << 3;
    return PA_OK;
}

} // namespace pa
