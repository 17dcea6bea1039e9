// Diagnostics.
//  * The bounded mbarrier wait every kernel of the library uses, exercised on
//    its own.  One warp initialises a barrier in shared memory and waits on its
//    first phase; unless told to arrive first, nothing completes that phase, so
//    the wait must give up after its time limit, record that in a device error
//    word and let the kernel return (the context stays usable).
//  * A read-only stream: every byte of a buffer read once with 16-byte
//    non-caching loads, the bandwidth ceiling of the decode kernels (which read
//    the cache and write almost nothing), for measuring them against it.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace pa {

__device__ uint32_t g_selftest_error; // bit 0: the diagnostic wait timed out

namespace {

__global__ void bounded_wait_kernel(uint64_t timeout_ns, int arrive_first)
{
    __shared__ __align__(8) uint64_t bar_storage;
    const uint32_t bar = ptx::smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && arrive_first)
        ptx::mbar_arrive(bar);
    __syncwarp();
    const bool ok = ptx::mbar_wait(bar, 0, timeout_ns);
    if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0)
        atomicOr(&g_selftest_error, 1u);
}

// Grid-stride read of n 16-byte vectors, four loads in flight per thread; the
// words are folded into one XOR per warp so the loads cannot be dropped.
__global__ void __launch_bounds__(512) stream_read_kernel(const uint4 *__restrict__ src, size_t n, uint32_t *sink)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
                    d = __ldcs(src + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
    }
    for (; i < n; i += stride) {
        const uint4 a = __ldcs(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    for (int o = 16; o > 0; o >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0)
        atomicXor(sink, acc);
}

} // namespace

int launch_stream_read(const void *src, size_t bytes, uint32_t *sink, void *stream)
{
    const size_t n = bytes / 16;
    if (n == 0)
        return PA_OK;
    int sms = 0;
    if (int rc = sm_count(&sms))
        return rc;
    stream_read_kernel<<<(unsigned)(4 * sms), 512, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(src), n, sink);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "stream read launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

int launch_selftest_wait(uint32_t timeout_us, int arrive_first, void *stream)
{
    bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)timeout_us * 1000u,
                                                                        arrive_first);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return PA_OK;
}

int read_selftest_error(uint32_t *code)
{
    uint32_t v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof v);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return fail(PA_ERR_CUDA, "reading self-test error word: %s", cudaGetErrorString(e));
    *code |= v << 4;
    return PA_OK;
}

} // namespace pa
