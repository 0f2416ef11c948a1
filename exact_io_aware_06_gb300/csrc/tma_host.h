// tma_host.h -- host-side creation of TMA tensor maps for [BH][N][d] tensors.
// cuTensorMapEncodeTiled is fetched through the runtime's driver-entry-point
// query, so the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tensor map over a dense [BH][N][d] tensor with elements of `elem_bytes`
// bytes, read in boxes of (box_x elements along d) x (box_y rows) x 1 head,
// 128-byte swizzled (box_x * elem_bytes must be 128).  Rows past N read as zero.
// Returns 0 on success.
inline int make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt,
                       uint32_t elem_bytes, uint64_t d, uint64_t N, uint64_t BH, uint32_t box_x,
                       uint32_t box_y) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return -1;
    cuuint64_t dims[3] = {d, N, BH};
    cuuint64_t strides[2] = {d * elem_bytes, N * d * elem_bytes};
    cuuint32_t box[3] = {box_x, box_y, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : static_cast<int>(r);
}

}  // namespace fa
