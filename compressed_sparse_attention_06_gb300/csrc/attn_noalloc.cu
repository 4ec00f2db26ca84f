// csa2_sparse_attn_noalloc: the sparse attention entry point for callers that are
// not allowed to allocate device memory.
//
// Some hosts of this library own every byte of device memory themselves: a
// serving engine that carves one arena out of the GPU at start-up and forbids its
// plugins from calling cudaMalloc, or a latency-critical loop where an allocation
// (and the synchronisation it may imply) is not acceptable.  Such callers cannot
// hand csa2_sparse_attn the workspace its key-split path wants.  This variant keeps
// that workspace in a fixed array compiled into the library instead, so the caller
// passes only its inputs and outputs.
//
// The array (CSA2_NOALLOC_SCRATCH_BYTES) is a file-scope device variable: every
// GPU that loads the library holds it until the process exits.  All calls share
// it, so calls whose kernels overlap on the GPU race on it.  Nothing in it has to
// start at zero: every call rewrites each partial result it later reads.
#include "attn_tc.cuh"
#include "csa2_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

// Device address of g_attn_scratch on the context's device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with that
// device current, once per context (the set-up of the first call), and kept in the
// context: it lives exactly as long as the context.  A device reset unloads the
// module and may move the array; the context (whose status word the reset frees as
// well) must then be destroyed and created again.
csa2_status scratch_address(csa2_ctx* ctx, void** out) {
    if (!ctx->noalloc_scratch) {
        int prev = 0;
        if (cudaGetDevice(&prev) != cudaSuccess) return CSA2_ERR_CUDA;
        if (prev != ctx->device && cudaSetDevice(ctx->device) != cudaSuccess) return CSA2_ERR_CUDA;
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (prev != ctx->device && cudaSetDevice(prev) != cudaSuccess) return CSA2_ERR_CUDA;
        if (e != cudaSuccess || !p) return CSA2_ERR_CUDA;
        ctx->noalloc_scratch = p;
    }
    *out = ctx->noalloc_scratch;
    return CSA2_OK;
}

}  // namespace

extern "C" csa2_status csa2_sparse_attn_noalloc(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const void* kv,
                                                csa2_dtype kv_dt, int64_t N, const int32_t* idx, int k,
                                                const void* swa, csa2_dtype swa_dt, int64_t swa_cap,
                                                int64_t swa_pos0, int window, const int64_t* q_pos,
                                                const float* sink, int B, int Q, int H, int c, float rope_base,
                                                unsigned flags, void* out, csa2_dtype out_dt, float* lse,
                                                void* stream) {
    if (!ctx) return CSA2_ERR_INVALID_ARG;
    // The CUDA-core key split must fit the fixed array; the tensor-core path is taken
    // only when its larger workspace fits as well.
    const size_t need = attn_simt_ws_bytes(ctx, B, Q, H, k, window);
    if (need > (size_t)CSA2_NOALLOC_SCRATCH_BYTES) return CSA2_ERR_INVALID_ARG;
    void* scratch = nullptr;
    csa2_status st = scratch_address(ctx, &scratch);
    if (st != CSA2_OK) return st;
    return csa2_sparse_attn(ctx, q, q_dt, kv, kv_dt, N, idx, k, swa, swa_dt, swa_cap, swa_pos0, window, q_pos, sink,
                            B, Q, H, c, rope_base, flags, out, out_dt, lse, scratch,
                            (size_t)CSA2_NOALLOC_SCRATCH_BYTES, stream);
}
