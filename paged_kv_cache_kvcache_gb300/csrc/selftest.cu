// Diagnostic: the bounded mbarrier wait every kernel of the library uses,
// exercised on its own.  One warp initialises a barrier in shared memory and
// waits on its first phase; unless told to arrive first, nothing completes
// that phase, so the wait must give up after its time limit, record that in a
// device error word and let the kernel return (the context stays usable).
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

} // namespace

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
