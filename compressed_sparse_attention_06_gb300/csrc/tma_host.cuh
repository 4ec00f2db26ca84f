// Host side of the tensor-memory-access (TMA) copies: the driver's tensor-map
// encoder, looked up once through the runtime (no link against libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

typedef CUresult (*Csa2EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static inline Csa2EncodeTiledFn csa2_encode_tiled_fn() {
    static Csa2EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<Csa2EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D map over `rows` bf16 rows of `cols` values (row stride cols * 2 bytes): box of
// box_cols x box_rows, 128-byte swizzle.
static inline bool csa2_make_bf16_map(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_cols,
                                      int box_rows) {
    Csa2EncodeTiledFn fn = csa2_encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over `rows` bf16 rows of 128 values, for copying `box_rows` rows whole: dims
// (64 values, rows, the two 64-value halves of a row) with strides 256 B (rows) and
// 128 B (halves); box 64 x box_rows x 2 with the 128-byte swizzle, so one copy lands
// the rows as [half][box_rows rows][64 values]: one K-chunk of 64 dims after the other,
// in 1 KB swizzle atoms of 8 rows.
static inline bool csa2_make_bf16_block_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
    Csa2EncodeTiledFn fn = csa2_encode_tiled_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
    cuuint64_t strides[2] = {256, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
