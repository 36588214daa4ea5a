// tensormap.cuh -- host-side TMA descriptor encoding shared by the kernels:
// the driver's cuTensorMapEncodeTiled is looked up once through the runtime
// (no link-time dependency on libcuda).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace fp8fg {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    // initialised once (thread-safe static initialisation)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        PFN_cuTensorMapEncodeTiled_v12000 f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        (void)cudaGetLastError();
        return f;
    }();
    return fn;
}

// 2-D row-major tensor [outer][inner] (row stride row_bytes) with a
// box_outer x box_inner box.  Out-of-range box elements read as zero.
inline int make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle) {
    auto fn = encode_tiled();
    if (fn == nullptr) return FP8_ERR_CUDA;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8fg
