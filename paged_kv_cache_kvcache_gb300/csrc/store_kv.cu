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
#include "ptx.cuh"
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

// INT8 prefill front end: the keys and values that a prefill batch attends over,
// dequantised into a bf16 scratch cache of 128-token blocks, each sequence's keys
// in consecutive blocks (the plan's scratch tables; scratch block sb holds keys
// e[1] .. e[1] + 127 of sequence e[0], e = scratch_items[sb]).  "面试问答准备:
// nano-vLLM 推理引擎优化", Q3, the prefill's dequantisation path: the values the
// block table references, read as code x token scale in fp32 and rounded to the
// model's dtype (bf16), feed the bf16 attention.  With `store`, the new tokens'
// rows (positions from the cached prefix on) are first quantised from k_in/v_in
// into the INT8 cache at their slots, as pa_store_kvcache_int8 does, and their
// scratch rows dequantise those codes and the stored fp16 scale, so the scratch
// holds what the cache then holds.
//
// Work unit: one (scratch row, tensor, KV head), handled by kThreadsPerRow<D>
// adjacent threads (32 values each): unit u is row u / (2 Hkv), then K heads, then
// V heads, so a warp reads and writes whole rows of K and of V (coalesced).  One
// unit per thread group; HBM-bound: 3 bytes moved per value (1 read, 2 written).
template <int D, bool kStore>
__global__ void __launch_bounds__(256) int8_gather_kernel(const GatherArgs a)
{
    constexpr int TPR = quant::kThreadsPerRow<D>;
    const uint32_t hkv = (uint32_t)a.num_kv_heads;
    const uint32_t j = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t unit = j / TPR;
    if (unit >= (uint32_t)a.scratch_blocks * 128u * 2u * hkv)
        return;
    const int h = (int)(j % TPR);
    const uint32_t r = unit / (2u * hkv); // scratch row
    const uint32_t c = unit - r * 2u * hkv;
    const bool is_v = c >= hkv;
    const int g = (int)(is_v ? c - hkv : c);
    const int4 e = __ldg(reinterpret_cast<const int4 *>(a.scratch_items) + 2 * (r >> 7));
    const int b = e.x, pos = e.y + (int)(r & 127), lk = e.z, cached = e.w;
    if (pos >= lk)
        return; // past the sequence end: the attention never reads this row's values
    uint32_t code[8];
    float sc;
    if (kStore && pos >= cached) {
        const int t = __ldg(a.scratch_items + 8 * (r >> 7) + 4) + pos; // packed row of the new token
        const int32_t slot = __ldg(a.slot_mapping + t);
        quant::RowPart part;
        quant::load_row_part((is_v ? a.v_in : a.k_in) + ((size_t)t * hkv + g) * D, h, part);
        const __half hs = __float2half_rn(quant::quantise_part<D>(part, code));
        if (slot >= 0 && slot < a.num_slots) {
            uint4 *dst = reinterpret_cast<uint4 *>((is_v ? a.v_codes_w : a.k_codes_w) + ((size_t)slot * hkv + g) * D +
                                                   32 * h);
            dst[0] = make_uint4(code[0], code[1], code[2], code[3]);
            dst[1] = make_uint4(code[4], code[5], code[6], code[7]);
            if (h == 0)
                (is_v ? a.v_scale_w : a.k_scale_w)[((size_t)(slot / a.block_size) * hkv + g) * a.block_size +
                                                   slot % a.block_size] = __half_as_ushort(hs);
        } else if (slot != -1 && !is_v && g == 0 && h == 0) {
            atomicOr(&g_store_error, 1u);
        }
        sc = __half2float(hs);
    } else {
        const int bs = a.block_size;
        const int blk = __ldg(a.block_tables + (size_t)b * a.max_blocks + pos / bs);
        const uint4 *src = reinterpret_cast<const uint4 *>((is_v ? a.v_codes : a.k_codes) +
                                                           (((size_t)blk * bs + pos % bs) * hkv + g) * D + 32 * h);
        const uint4 x0 = __ldcs(src), x1 = __ldcs(src + 1);
        sc = __half2float(__ushort_as_half(__ldg((is_v ? a.v_scale : a.k_scale) + ((size_t)blk * hkv + g) * bs + pos % bs)));
        code[0] = x0.x, code[1] = x0.y, code[2] = x0.z, code[3] = x0.w;
        code[4] = x1.x, code[5] = x1.y, code[6] = x1.z, code[7] = x1.w;
    }
    uint4 o[4];
    quant::dequantise_part(code, sc, o);
    uint16_t *out = (is_v ? a.v_out : a.k_out) + ((size_t)r * hkv + g) * D + 32 * h;
    if (a.out_v8) { // 32-byte stores: half the store instructions (the gather is bound by them)
        ptx::st_global_v8(out, o[0].x, o[0].y, o[0].z, o[0].w, o[1].x, o[1].y, o[1].z, o[1].w);
        ptx::st_global_v8(out + 16, o[2].x, o[2].y, o[2].z, o[2].w, o[3].x, o[3].y, o[3].z, o[3].w);
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(out);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = o[i];
    }
}

int launch_int8_gather(const GatherArgs &a, void *stream)
{
    const int threads = 256;
    const int64_t n = (int64_t)a.scratch_blocks * 128 * 2 * a.num_kv_heads * (a.head_dim / 32);
    if (n == 0)
        return PA_OK;
    if (n > INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED, "INT8 prefill scratch of %lld (row, tensor, head) units exceeds int32",
                    (long long)(n / (a.head_dim / 32)));
    const bool st = a.k_in != nullptr;
    auto kern = a.head_dim == 128 ? (st ? int8_gather_kernel<128, true> : int8_gather_kernel<128, false>)
                                  : (st ? int8_gather_kernel<64, true> : int8_gather_kernel<64, false>);
    kern<<<(unsigned)((n + threads - 1) / threads), threads, 0, (cudaStream_t)stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "int8 gather launch: %s", cudaGetErrorString(e));
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
