// tma_host.cuh -- host-side creation of TMA tensor maps through the driver's
// cuTensorMapEncodeTiled, looked up at run time (the library does not link
// libcuda, so it loads on machines without a GPU driver).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace gdr {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D BF16 tensor [d2][d1][d0] (d0 contiguous) with byte strides s1 (dim 1)
// and s2 (dim 2); box {b0, b1, b2}; 128-byte swizzle; out-of-range elements
// read as zero.  Returns false if the driver rejects the map.
inline bool make_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                              uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
                              uint32_t b2) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D BF16 tensor [d1][d0] (d0 contiguous), byte stride s1; box {b0, b1};
// 128-byte swizzle; out-of-range elements read as zero.
inline bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                              uint64_t s1, uint32_t b0, uint32_t b1) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {s1};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gdr
