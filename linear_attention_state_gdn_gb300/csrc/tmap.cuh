// tmap.cuh -- host-side construction of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query, so the library does not link libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <mutex>

namespace hypic {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tiled map over a row-major 2D array [rows][cols] (row pitch `pitch` bytes), box
// [box_rows][box_cols].
inline bool make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint64_t cols,
                         uint64_t rows, uint64_t pitch, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle sw) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiled map over a row-major 3D array [d2][d1][d0] (pitches in bytes), box [b2][b1][b0].
inline bool make_tmap_3d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint64_t d0,
                         uint64_t d1, uint64_t d2, uint64_t pitch1, uint64_t pitch2, uint32_t b0,
                         uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {pitch1, pitch2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace hypic
