// Block copy for copy-on-write forks of shared cache blocks.
//
// Source: "vLLM / SGLang 面试源码深挖", section 4 (beam search and KV block
// fork), the follow-up on a native block-table fork: parent and child first
// share block ids; when an append would land in a shared, still-mutable last
// block, the child gets a new block and the valid KV of the shared block is
// copied into it, after which each writes its own.  Also "推理系统"
// (PagedAttention paragraph): shared blocks are copied on write, as in fork.
//
// Each (src, dst, n) triple copies cache rows src*bs + i -> dst*bs + i for
// i < n, in K and in V (and, for an INT8 cache, the rows' scales).  Grid:
// (triple, 16-row chunk); 16-byte vectors.
#include <cuda_runtime.h>

#include "internal.h"

namespace pa {

__device__ uint32_t g_copy_error; // 1 = a triple outside the pool was skipped

// INT8 caches (k_scale != NULL): codes move like bf16 rows (row_vecs counts
// their 16-byte vectors) and the first chunk's CTA also moves each KV head's
// run of n fp16 scales, [src][g][0..n) -> [dst][g][0..n).
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                                          const int3 *__restrict__ triples, int32_t row_vecs,
                                                          int32_t block_size, int32_t num_blocks,
                                                          uint16_t *__restrict__ k_scale,
                                                          uint16_t *__restrict__ v_scale, int32_t num_kv_heads)
{
    const int3 tr = triples[blockIdx.x];
    const int src = tr.x, dst = tr.y, n = tr.z;
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || n < 0 || n > block_size) {
        if (threadIdx.x == 0)
            atomicOr(&g_copy_error, 1u);
        return;
    }
    if (k_scale && blockIdx.y == 0) {
        for (int i = threadIdx.x; i < num_kv_heads * n; i += blockDim.x) {
            const int h = i / n, r = i % n;
            const size_t from = ((size_t)src * num_kv_heads + h) * block_size + r;
            const size_t to = ((size_t)dst * num_kv_heads + h) * block_size + r;
            const uint16_t a = k_scale[from], b = v_scale[from];
            k_scale[to] = a;
            v_scale[to] = b;
        }
    }
    const int r0 = blockIdx.y * 16;
    const int rows = min(16, n - r0);
    if (rows <= 0)
        return;
    const size_t s = ((size_t)src * block_size + r0) * row_vecs;
    const size_t d = ((size_t)dst * block_size + r0) * row_vecs;
    const int total = rows * row_vecs;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const uint4 a = k_cache[s + i];
        const uint4 b = v_cache[s + i];
        k_cache[d + i] = a;
        v_cache[d + i] = b;
    }
}

int launch_copy_blocks(const pa_dims &dm, void *k_cache, void *v_cache, const int32_t *triples, int32_t n,
                       void *stream, void *k_scale, void *v_scale)
{
    const int elem = k_scale ? 1 : 2; // INT8 codes or bf16 values
    const int32_t row_vecs = dm.num_kv_heads * dm.head_dim * elem / 16;
    dim3 grid((unsigned)n, (unsigned)((dm.block_size + 15) / 16));
    copy_blocks_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), reinterpret_cast<const int3 *>(triples),
        row_vecs, dm.block_size, dm.num_blocks, static_cast<uint16_t *>(k_scale), static_cast<uint16_t *>(v_scale),
        dm.num_kv_heads);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "copy_blocks launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

int read_copy_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_copy_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_copy_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading copy error word: %s", cudaGetErrorString(e));
    *code |= v << 2;
    return PA_OK;
}

} // namespace pa
