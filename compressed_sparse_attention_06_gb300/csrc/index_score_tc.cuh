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
// Same contract as index_score_tc_dispatch.  With q_bf16 (bf16 [B, Q, 64, 128]) the
// queries are packed to MXFP4 inside the scan (q_idx unused) and, if q_mx_out is not
// NULL, written there too.
csa2_status index_score_fp4_dispatch(csa2_ctx* ctx, const void* q_idx, const float* w, const void* k_idx, int B,
                                     int Q, int64_t N, int H_I, const int64_t* n_visible, const int32_t* pool,
                                     int n_pool, int block, float* scores, float* block_max, uint32_t* hist,
                                     cudaStream_t s, const void* q_bf16 = nullptr, uint8_t* q_mx_out = nullptr);
// hist != NULL: the scan adds every visible block maximum's first radix digit to
// hist ([B*Q, CSA2_BLOCK_HIST_BINS], zeroed beforehand).  The other scans leave it
// to block_hist_from_max (select.cu).

// Pool histogram helpers (select.cu): zero rows x CSA2_BLOCK_HIST_BINS words; count
// the first radix digit of the visible block maxima of each row (n_visible entries
// per row, blocks of `block`).
csa2_status block_hist_zero(uint32_t* hist, int64_t rows, cudaStream_t s);
csa2_status block_hist_from_max(const float* bmax, int64_t rows, int64_t ld, const int64_t* n_visible, int block,
                                uint32_t* hist, cudaStream_t s);
