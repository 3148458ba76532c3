// tma_map.h -- host-side TMA descriptors for [rows, heads, d] bf16 tensors,
// shared by the attention kernels' launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pva {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// [rows, heads, d] bf16 (elem_bytes = 2) or fp32 (4) viewed as a 3-D tensor
// (d, heads, rows); boxes of box_rows rows x 128 bytes (64 bf16 or 32 fp32
// elements) with 128-byte swizzle; rows past the end read as zero (loads) or
// are not written (stores).
inline bool make_map(CUtensorMap* m, const void* ptr, int32_t rows, int32_t heads, int32_t d,
                     uint32_t box_rows = 128, int elem_bytes = 2) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)heads * d * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), 1, box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m,
               elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
               3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pva
