// TMA tensor-map encoding shared by the kernels that load through TMA.  The
// driver's cuTensorMapEncodeTiled is looked up once through the runtime (no
// link against libcuda).
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace pa {

static PFN_cuTensorMapEncodeTiled_v12000 lookup_encoder()
{
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    cudaGetLastError();
    return nullptr;
}

int encode_tmap_3d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t d0, uint64_t d1,
                   uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                   CUtensorMapSwizzle swizzle, const char *what)
{
    static const PFN_cuTensorMapEncodeTiled_v12000 enc = lookup_encoder();
    if (!enc)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, type, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
    return PA_OK;
}

} // namespace pa
