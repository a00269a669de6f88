// tmap.cu -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled, fetched once from
// the driver through the runtime so that the library has no link-time dependency on libcuda).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace mla {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;

void init_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_init_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (g_init_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
        g_init_err = cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        bool swizzle128) {
    std::call_once(g_once, init_encode);
    if (g_init_err != cudaSuccess) return g_init_err;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = g_encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mla
