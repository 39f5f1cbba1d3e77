// Host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point so that the library does not link
// libcuda directly).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

namespace moe {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return nullptr;
    }();
    return fn;
}

// 2D row-major [rows, cols] of `esize`-byte elements with a (box_rows x
// box_cols) box; reads outside the tensor return zeros.
inline bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dtype, uint32_t esize, const void *base, uint64_t rows,
                         uint64_t cols, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swz) {
    auto fn = tmap_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 [rows, cols]: operand loads use 64-column (128-byte) boxes with
// 128-byte swizzle.
inline bool make_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      uint32_t box_cols = 64, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, cols, box_rows, box_cols, swz);
}

// Byte matrix (E4M3 codes) [rows, cols]: 128-byte boxes, 128-byte swizzle.
inline bool make_tmap_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, box_rows, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace moe
