// Host-side helpers for TMA tensor maps (driver entry point resolved through the runtime,
// so the library does not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lla {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D fp16 tensor [slices][rows][inner] (inner contiguous), box [1][box_rows][64], 128-byte
// swizzle, zero fill outside the tensor.  Returns false if the encoder is unavailable or
// rejects the arguments.
inline bool make_tmap_f16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t slices,
                             uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, rows, slices};
    cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D 16-bit tensor [slices][rows][inner] (inner contiguous) whose slices lie slice_rows >= rows
// rows apart: rows past `rows` of a slice read as zeros, never as the memory behind them.  Box
// [1][box_rows][64], 128-byte swizzle.  type: CU_TENSOR_MAP_DATA_TYPE_FLOAT16 or _BFLOAT16.
inline bool make_tmap_16b_3d_strided(CUtensorMap* map, const void* base, CUtensorMapDataType type, uint64_t inner,
                                     uint64_t rows, uint64_t slices, uint64_t slice_rows, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc || slice_rows < rows) return false;
    cuuint64_t dims[3] = {inner, rows, slices};
    cuuint64_t strides[2] = {inner * 2, inner * slice_rows * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace lla
