// Tensor-core Lightning-indexer scan (tcgen05).  Not built yet: every shape is
// reported unsupported so csa2_index_score runs its CUDA-core kernel.
#include "index_score_tc.cuh"

csa2_status index_score_tc_dispatch(csa2_ctx*, const void*, const float*, const void*, csa2_dtype, int, int,
                                    int64_t, int, const int64_t*, const int32_t*, int, int, float*, float*,
                                    cudaStream_t) {
    return CSA2_ERR_UNSUPPORTED;
}
