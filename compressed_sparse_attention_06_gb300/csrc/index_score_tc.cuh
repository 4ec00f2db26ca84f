// Tensor-core (tcgen05) Lightning-indexer scan: dispatch entry used by
// csa2_index_score.  Returns CSA2_ERR_UNSUPPORTED when the shape is not covered,
// in which case the CUDA-core kernel runs.
#pragma once
#include "csa2_internal.cuh"

csa2_status index_score_tc_dispatch(csa2_ctx* ctx, const void* q_idx, const float* w, const void* k_idx,
                                    csa2_dtype k_dt, int B, int Q, int64_t N, int H_I,
                                    const int64_t* n_visible, const int32_t* pool, int n_pool, int block,
                                    float* scores, float* block_max, cudaStream_t s);

// FP4 QK path (tcgen05 kind::mxf4): MXFP4 queries [B, Q, 64, 68] over MXFP4 keys.
// Same contract as index_score_tc_dispatch.
csa2_status index_score_fp4_dispatch(csa2_ctx* ctx, const void* q_idx, const float* w, const void* k_idx, int B,
                                     int Q, int64_t N, int H_I, const int64_t* n_visible, const int32_t* pool,
                                     int n_pool, int block, float* scores, float* block_max, cudaStream_t s);
