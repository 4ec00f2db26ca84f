// Context, status word and status strings of the CSA2 C ABI.
#include <new>

#include "csa2_internal.cuh"

extern "C" const char* csa2_status_string(csa2_status s) {
    switch (s) {
        case CSA2_OK: return "ok";
        case CSA2_ERR_INVALID_ARG: return "invalid argument (nothing launched)";
        case CSA2_ERR_UNSUPPORTED: return "unsupported dtype or shape combination";
        case CSA2_ERR_CUDA: return "CUDA runtime or launch error";
        case CSA2_ERR_TIMEOUT: return "a device-side bounded wait expired";
        case CSA2_ERR_DEVICE: return "a kernel met an out-of-range index";
    }
    return "unknown status";
}

extern "C" int csa2_version(void) { return 1; }

extern "C" csa2_status csa2_ctx_create(int device, csa2_ctx** out) {
    if (!out) return CSA2_ERR_INVALID_ARG;
    *out = nullptr;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) return CSA2_ERR_CUDA;
    if (device < 0 || device >= n) return CSA2_ERR_INVALID_ARG;
    int prev = 0;
    CSA2_CHECK_CUDA(cudaGetDevice(&prev));
    CSA2_CHECK_CUDA(cudaSetDevice(device));
    csa2_ctx* c = new (std::nothrow) csa2_ctx;
    if (!c) return CSA2_ERR_CUDA;
    c->device = device;
    c->status = nullptr;
    c->num_sms = 0;
    c->stall_next = 0;
    c->stall_budget = 0;
    c->cluster16 = -1;
    c->noalloc_scratch = nullptr;
    cudaError_t e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaMalloc(&c->status, sizeof(unsigned int));
    if (e == cudaSuccess) e = cudaMemset(c->status, 0, sizeof(unsigned int));
    cudaSetDevice(prev);
    if (e != cudaSuccess) {
        if (c->status) cudaFree(c->status);
        delete c;
        return CSA2_ERR_CUDA;
    }
    *out = c;
    return CSA2_OK;
}

extern "C" csa2_status csa2_ctx_destroy(csa2_ctx* ctx) {
    if (!ctx) return CSA2_ERR_INVALID_ARG;
    if (ctx->status) cudaFree(ctx->status);
    delete ctx;
    return CSA2_OK;
}

extern "C" csa2_status csa2_ctx_check(csa2_ctx* ctx, void* stream) {
    if (!ctx) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return CSA2_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, ctx->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA2_ERR_CUDA;
    if (word) {
        if (cudaMemset(ctx->status, 0, sizeof(word)) != cudaSuccess) return CSA2_ERR_CUDA;
    }
    if (word & CSA2_DEVBIT_TIMEOUT) return CSA2_ERR_TIMEOUT;
    if (word & CSA2_DEVBIT_RANGE) return CSA2_ERR_DEVICE;
    return CSA2_OK;
}

extern "C" csa2_status csa2_ctx_test_stall_next(csa2_ctx* ctx, long long budget_cycles) {
    if (!ctx || budget_cycles < 0) return CSA2_ERR_INVALID_ARG;
    ctx->stall_next = 1;
    ctx->stall_budget = budget_cycles;
    return CSA2_OK;
}
