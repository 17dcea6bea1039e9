// Batched single-token GQA decode over the paged KV cache, split-KV + LSE combine.
//
// Sources (page title, section):
//  - "手搓 vLLM 推理引擎" (LLM-101-CN nano-vllm walkthrough), Step 4: decode
//    attends one new query per sequence to all context_lens[b] cached keys,
//    found through the sequence's block table.
//  - "推理系统" (CS 与 LLM 学习知识库), "瓶颈不是算力，是带宽": decode
//    attention does ~1 flop per byte of K/V read, so its time is the bytes
//    read divided by the memory bandwidth.
//  - "面试问答准备: nano-vLLM 推理引擎优化", Q3 follow-ups / summary table:
//    Paged Attention v2 reuses each KV head for its whole query-head group and
//    uses tensor cores; Split-K cuts a long context into segments that each
//    emit a local max, normaliser and fp32 accumulator, merged by a second
//    kernel with log-sum-exp.
//
// GB300 design.  One CTA per (work item = sequence x key range, KV head); its
// 4 warps stream disjoint 16-token chunks of K and V for that head through a
// 3-stage cp.async (16-byte, L2-only) pipeline into XOR-swizzled shared
// memory.  The G query heads of the group share every K/V byte read:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T      (mma.sync m16n8k16, bf16)
//   O^T[D x 8 heads]    += V^T[D x 16] . P^T      (P^T via movmatrix.trans)
// so the per-byte arithmetic (G flops/byte at G = 7) runs on the tensor pipe
// instead of the FP32 lanes, and the kernel stays bound by HBM.  Online
// softmax state lives in the accumulator fragments' own threads (no shuffles
// except one 3-step max per chunk).  The 4 warps merge through shared memory;
// a single-split sequence writes bf16 directly, otherwise (o/l, log2-sum-exp)
// partials go to the workspace and a combine kernel merges them.
#include <mutex>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecLayout {
    static constexpr int kRowBytes = D * 2;             // one head row of one token
    static constexpr int kChunkBytes = 16 * kRowBytes;  // 16 tokens of K (or V)
    static constexpr int kStageBytes = 2 * kChunkBytes; // K + V
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kSmemBytes = kWarps * kWarpBytes;
    static constexpr int kVecPerRow = D / 8;            // 16-byte vectors per row
};

struct DecParams {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
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
    // fused store (FUSED kernels only): the new token's K/V rows, its slot, the context lengths
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    __nv_bfloat16 *k_store;
    __nv_bfloat16 *v_store;
    const int32_t *slot_mapping;
    const int32_t *context_lens;
    int64_t num_slots;
};

__device__ uint32_t g_fused_error; // bit 0: a fused-store slot outside [-1, num_slots) was skipped

// FUSED: the CTA whose work item ends at the sequence's last key (the token
// being decoded) writes that token's K/V rows into the cache slot and takes
// its key from the input instead of the cache, so store and attention need
// no ordering between launches.
template <int D, int NT, bool FUSED>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_split_kernel(const DecParams p)
{
    using L = DecLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int4 item = p.items[blockIdx.x / p.num_kv_heads];
    const int b = item.x, k0 = item.y, pslot = item.w;
    const int g = blockIdx.x % p.num_kv_heads;
    const int G = p.group;
    const int Hq = p.num_heads;
    // FUSED: does this item hold the new token (the last key)?  Then the cache supplies keys k0 .. ctx-2.
    const bool has_new = FUSED && item.z > 0 && item.z == __ldg(p.context_lens + b);
    const int k1 = has_new ? item.z - 1 : item.z;

    // Q^T fragments: B operand (k = d, n = head) of the score MMA.
    uint32_t qf[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hl = nt * 8 + (lane >> 2);
        const bool valid = hl < G;
        const uint32_t *qrow =
            reinterpret_cast<const uint32_t *>(p.q + ((size_t)b * Hq + (size_t)g * G + (valid ? hl : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[nt][kk][0] = valid ? __ldg(qrow + kk * 8 + (lane & 3)) : 0u;
            qf[nt][kk][1] = valid ? __ldg(qrow + kk * 8 + 4 + (lane & 3)) : 0u;
        }
    }

    const int nchunks = (k1 - k0 + 15) >> 4;
    const int my_n = nchunks > warp ? (nchunks - warp + kWarps - 1) / kWarps : 0;
    const uint32_t wbase = ptx::smem_u32(smem) + warp * L::kWarpBytes;
    const int32_t *bt_row = p.block_tables + (size_t)b * p.max_blocks;
    const int bs = p.block_size;
    const int Hkv = p.num_kv_heads;
    int blk_cache = 0;

    auto issue = [&](int i) {
        if ((i & 31) == 0) { // refresh the block ids of local chunks i .. i+31, one per lane
            const int key = k0 + 16 * (warp + kWarps * (i + lane));
            blk_cache = key < k1 ? __ldg(bt_row + key / bs) : 0;
        }
        const int phys = __shfl_sync(0xffffffffu, blk_cache, i & 31);
        const int key0 = k0 + 16 * (warp + kWarps * i);
        const int64_t row0 = (int64_t)phys * bs + (key0 & (bs - 1));
        const uint32_t sbase = wbase + (i % kStages) * L::kStageBytes;
#pragma unroll
        for (int r = 0; r < L::kVecPerRow / 2; ++r) {
            const int e = r * 32 + lane;
            const int t = e / L::kVecPerRow;
            const int c = e % L::kVecPerRow;
            const bool valid = key0 + t < k1;
            const size_t off = ((size_t)(row0 + t) * Hkv + g) * D + c * 8;
            const uint32_t dst = sbase + t * L::kRowBytes + ((c ^ (t & 7)) << 4);
            ptx::cp_async_16(dst, valid ? (const void *)(p.k_cache + off) : (const void *)p.k_cache, valid ? 16u : 0u);
            ptx::cp_async_16(dst + L::kChunkBytes, valid ? (const void *)(p.v_cache + off) : (const void *)p.v_cache,
                             valid ? 16u : 0u);
        }
    };

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

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < my_n)
            issue(s);
        ptx::cp_async_commit();
    }

    // ldmatrix row addressing (per lane) inside a 16-token chunk
    const int a_tok = (lane & 7) + ((lane >> 3) & 1) * 8; // K: A = K[tok][d]
    const int a_hi = lane >> 4;
    const int v_tok = (lane & 7) + (lane >> 4) * 8;       // V: A = V^T via .trans
    const int v_hi = (lane >> 3) & 1;

    for (int i = 0; i < my_n; ++i) {
        __syncwarp();
        if (i + kStages - 1 < my_n)
            issue(i + kStages - 1);
        ptx::cp_async_commit();
        ptx::cp_async_wait<kStages - 1>();
        __syncwarp();

        const uint32_t kb = wbase + (i % kStages) * L::kStageBytes;
        const uint32_t vb = kb + L::kChunkBytes;
        const int key0 = k0 + 16 * (warp + kWarps * i);

        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            const int c = 2 * kk + a_hi;
            ptx::ldmatrix_x4(kb + a_tok * L::kRowBytes + ((c ^ (a_tok & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                ptx::mma_16816(sc[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
        }

        const bool v0 = key0 + (lane >> 2) < k1;
        const bool v1 = key0 + (lane >> 2) + 8 < k1;
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float s0 = v0 ? sc[nt][0] * p.scale_log2 : -INFINITY;
            const float s1 = v0 ? sc[nt][1] * p.scale_log2 : -INFINITY;
            const float s2 = v1 ? sc[nt][2] * p.scale_log2 : -INFINITY;
            const float s3 = v1 ? sc[nt][3] * p.scale_log2 : -INFINITY;
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
#pragma unroll
            for (int mi = 0; mi < D / 16; ++mi) {
                acc[nt][mi][0] *= al0;
                acc[nt][mi][1] *= al1;
                acc[nt][mi][2] *= al0;
                acc[nt][mi][3] *= al1;
            }
            pb[nt][0] = ptx::movmatrix_trans(ptx::pack_bf16(p0, p1));
            pb[nt][1] = ptx::movmatrix_trans(ptx::pack_bf16(p2, p3));
        }

#pragma unroll
        for (int mi = 0; mi < D / 16; ++mi) {
            uint32_t a0, a1, a2, a3;
            const int c = 2 * mi + v_hi;
            ptx::ldmatrix_x4_trans(vb + v_tok * L::kRowBytes + ((c ^ (v_tok & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                ptx::mma_16816(acc[nt][mi], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
        }
    }
    ptx::cp_async_wait<0>();

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
    float *mrg_m = reinterpret_cast<float *>(smem);
    float *mrg_l = mrg_m + kWarps * H8;
    float *mrg_o = mrg_l + kWarps * H8; // [warp][head][D]
    float *s_new = mrg_o + (size_t)kWarps * H8 * D; // FUSED: the new key's score per head (log2 units)
    if constexpr (FUSED) {
        if (has_new) {
            const size_t row = ((size_t)b * p.num_kv_heads + g) * D;
            // the new key's score for each head of the group: one warp per head, D/32 values per lane
            for (int hl = warp; hl < G; hl += kWarps) {
                const __nv_bfloat16 *qr = p.q + ((size_t)b * Hq + (size_t)g * G + hl) * D;
                float acc_s = 0.f;
#pragma unroll
                for (int e = 0; e < D / 32; ++e)
                    acc_s += __bfloat162float(qr[lane + 32 * e]) * __bfloat162float(p.k_new[row + lane + 32 * e]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    acc_s += __shfl_xor_sync(0xffffffffu, acc_s, o);
                if (lane == 0)
                    s_new[hl] = acc_s * p.scale_log2;
            }
            // the store: this head's K and V rows of the new token into its slot
            const int32_t slot = __ldg(p.slot_mapping + b);
            if (slot >= 0 && slot < p.num_slots) {
                const size_t dst = ((size_t)slot * p.num_kv_heads + g) * D;
                for (int i = threadIdx.x; i < 2 * (D / 8); i += blockDim.x) {
                    const bool isv = i >= D / 8;
                    const int c = isv ? i - D / 8 : i;
                    const uint4 v = *reinterpret_cast<const uint4 *>((isv ? p.v_new : p.k_new) + row + 8 * c);
                    *reinterpret_cast<uint4 *>((isv ? p.v_store : p.k_store) + dst + 8 * c) = v;
                }
            } else if (slot != -1 && threadIdx.x == 0) {
                atomicOr(&g_fused_error, 1u);
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int h0 = nt * 8 + (lane & 3) * 2;
        if (lane < 4) {
            mrg_m[warp * H8 + h0] = m_r[nt][0];
            mrg_m[warp * H8 + h0 + 1] = m_r[nt][1];
            mrg_l[warp * H8 + h0] = l_r[nt][0];
            mrg_l[warp * H8 + h0 + 1] = l_r[nt][1];
        }
#pragma unroll
        for (int mi = 0; mi < D / 16; ++mi) {
            const int d = mi * 16 + (lane >> 2);
            float *o0 = mrg_o + ((size_t)warp * H8 + h0) * D;
            float *o1 = o0 + D;
            o0[d] = acc[nt][mi][0];
            o1[d] = acc[nt][mi][1];
            o0[d + 8] = acc[nt][mi][2];
            o1[d + 8] = acc[nt][mi][3];
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
                O += f * mrg_o[((size_t)w * H8 + hl) * D + d];
            }
            if (FUSED && has_new) { // the new token: weight 2^(s - M), value from the input row
                const float f = ptx::ex2(s_new[hl] - M);
                Lsum += f;
                O += f * __bfloat162float(p.v_new[((size_t)b * p.num_kv_heads + g) * D + d]);
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

// out[b][h] = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M), over the splits of sequence b.
// One warp per (sequence, head), D/32 values per lane.  The splits' partials are
// loaded kBatch at a time before any is used (a split's loads would otherwise wait
// for the previous split's), and accumulated in split order.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const float *__restrict__ part_o,
                                                             const float *__restrict__ part_lse,
                                                             const int32_t *__restrict__ seq_items,
                                                             __nv_bfloat16 *__restrict__ out, int num_heads)
{
    constexpr int E = D / 32;
    constexpr int kBatch = 8;
    using Vec = typename std::conditional<E == 4, float4, float2>::type;
    const int b = blockIdx.x;
    const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int s0 = seq_items[b], n = seq_items[b + 1] - s0;
    if (n <= 1 || h >= num_heads)
        return;
    const float *lse = part_lse + (size_t)s0 * num_heads + h;
    const float *po = part_o + ((size_t)s0 * num_heads + h) * D + lane * E;
    const size_t o_stride = (size_t)num_heads * D;
    float M = -INFINITY;
    for (int s = 0; s < n; ++s)
        M = fmaxf(M, __ldg(lse + (size_t)s * num_heads));
    float accv[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        accv[e] = 0.f;
    float W = 0.f;
    for (int s = 0; s < n; s += kBatch) {
        float l[kBatch];
        Vec o[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (s + i < n) {
                l[i] = __ldg(lse + (size_t)(s + i) * num_heads);
                o[i] = __ldg(reinterpret_cast<const Vec *>(po + (size_t)(s + i) * o_stride));
            }
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (s + i < n) {
                const float w = l[i] == -INFINITY ? 0.f : ptx::ex2(l[i] - M);
                W += w;
                const float *v = reinterpret_cast<const float *>(&o[i]);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    accv[e] += w * v[e];
            }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __nv_bfloat16 *dst = out + ((size_t)b * num_heads + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e)
        dst[e] = __float2bfloat16_rn(accv[e] * inv);
}

template <int D, int NT, bool FUSED>
int launch_split(const DecodeArgs &a, const DecParams &p, cudaStream_t stream)
{
    if (int rc = ensure_smem<decode_split_kernel<D, NT, FUSED>>(DecLayout<D>::kSmemBytes, "decode"))
        return rc;
    // flat grid, heads of one work item adjacent: they read neighbouring
    // segments of the same token rows at about the same time (DRAM locality)
    dim3 grid((unsigned)(a.num_items * a.dims.num_kv_heads));
    decode_split_kernel<D, NT, FUSED><<<grid, kWarps * 32, DecLayout<D>::kSmemBytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return launch_decode_combine(a, stream);
}

template <int D, int NT>
int occupancy()
{
    int n = 0;
    cudaFuncSetAttribute(decode_split_kernel<D, NT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         DecLayout<D>::kSmemBytes);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<D, NT, false>, kWarps * 32,
                                                      DecLayout<D>::kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return 2;
    }
    return n;
}

} // namespace

int launch_decode_combine(const DecodeArgs &a, void *stream)
{
    if (!a.part_o)
        return PA_OK;
    dim3 cg((unsigned)a.num_seqs, (unsigned)((a.dims.num_heads + 3) / 4));
    auto kern = a.dims.head_dim == 128 ? decode_combine_kernel<128> : decode_combine_kernel<64>;
    kern<<<cg, 128, 0, static_cast<cudaStream_t>(stream)>>>(a.part_o, a.part_lse, a.seq_items,
                                                            static_cast<__nv_bfloat16 *>(a.out), a.dims.num_heads);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "decode combine launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

int launch_decode(const DecodeArgs &a, void *stream)
{
    DecParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k_cache = static_cast<const __nv_bfloat16 *>(a.k_cache);
    p.v_cache = static_cast<const __nv_bfloat16 *>(a.v_cache);
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
    if (a.k_new) { // fused store + decode
        p.k_new = static_cast<const __nv_bfloat16 *>(a.k_new);
        p.v_new = static_cast<const __nv_bfloat16 *>(a.v_new);
        p.k_store = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.k_cache));
        p.v_store = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.v_cache));
        p.slot_mapping = a.slot_mapping;
        p.context_lens = a.context_lens;
        p.num_slots = (int64_t)a.dims.num_blocks * a.dims.block_size;
        if (a.dims.head_dim == 128)
            return two ? launch_split<128, 2, true>(a, p, s) : launch_split<128, 1, true>(a, p, s);
        return two ? launch_split<64, 2, true>(a, p, s) : launch_split<64, 1, true>(a, p, s);
    }
    if (a.dims.head_dim == 128)
        return two ? launch_split<128, 2, false>(a, p, s) : launch_split<128, 1, false>(a, p, s);
    return two ? launch_split<64, 2, false>(a, p, s) : launch_split<64, 1, false>(a, p, s);
}

int read_fused_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fused_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_fused_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading fused-store error word: %s", cudaGetErrorString(e));
    *code |= v; // same meaning as the store kernel's bit 0
    return PA_OK;
}

// Library-owned decode scratch for pa_decode_static (callers that cannot
// allocate).  Held by every device that loads the library until exit.
static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_STATIC_SCRATCH_BYTES];

int decode_static_scratch(void **ptr)
{
    // one lookup per device, made with that device current
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PA_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess)
            return fail(PA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return PA_OK;
}

int decode_ctas_per_sm(int head_dim, int group)
{
    const bool two = group > 8;
    if (head_dim == 128)
        return two ? occupancy<128, 2>() : occupancy<128, 1>();
    return two ? occupancy<64, 2>() : occupancy<64, 1>();
}

} // namespace pa
