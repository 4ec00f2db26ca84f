// Lightning-indexer scores (DSA-to-CSA/HCA page eq. (16)):
//     I[t, s] = sum_h w[t, h] * ReLU(q^I[t, h] . K^I[s])
// over the entries visible to the query (s < n_visible), with the block maximum
// over `block` consecutive entries fused into the epilogue (CSA2 page,
// «解码器里的分层索引»), or over the pooled candidates of a Reindex layer.
//
// This file holds the CUDA-core kernel: one thread per entry, the entry's key row
// in registers, the query's H_I x 128 indexer heads in shared memory (read as
// warp-wide broadcasts), fp32 FMA over exact bf16 / FP4 products.  It serves f32
// inputs, the shapes the tensor-core scans do not cover, and is the reference point
// for them.  MXFP4 queries are dequantised into shared memory.
#include <type_traits>

#include <algorithm>

#include "csa2_internal.cuh"
#include "index_score_tc.cuh"

namespace {

constexpr int D_IDX = 128;
constexpr int SIMT_TILE = 128;

enum KFmt { K_F32 = 0, K_BF16 = 1, K_MX = 2 };

template <int KF>
__device__ __forceinline__ void load_key_row(const void* kI, int64_t row, float (&k)[D_IDX]) {
    if (KF == K_F32) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(kI) + row * D_IDX);
#pragma unroll
        for (int i = 0; i < D_IDX / 4; ++i) {
            float4 v = p[i];
            k[4 * i] = v.x; k[4 * i + 1] = v.y; k[4 * i + 2] = v.z; k[4 * i + 3] = v.w;
        }
    } else if (KF == K_BF16) {
        const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(kI) + row * D_IDX);
#pragma unroll
        for (int i = 0; i < D_IDX / 8; ++i) {
            uint4 v = p[i];
            uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                k[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
                k[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
            }
        }
    } else {
        const uint32_t* p = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(kI) +
                                                              row * mxfp4_row_bytes(D_IDX));
        uint32_t sw = p[D_IDX / 8];   // 4 scale bytes after 64 code bytes
        float sc[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) sc[g] = e8m0_to_f32((sw >> (8 * g)) & 0xFF);
#pragma unroll
        for (int i = 0; i < D_IDX / 8; ++i) {
            uint32_t v = p[i];
#pragma unroll
            for (int j = 0; j < 8; ++j) k[8 * i + j] = e2m1_to_f32((v >> (4 * j)) & 0xF) * sc[(8 * i) / 32];
        }
    }
}

struct QMx {};   // query tag: MXFP4 rows of 68 bytes per head

template <typename TQ>
__device__ __forceinline__ void load_queries(const void* qI, int64_t bq, int H_I, float* qs) {
    if constexpr (std::is_same<TQ, QMx>::value) {
        const uint8_t* q8 = reinterpret_cast<const uint8_t*>(qI) + bq * (int64_t)H_I * mxfp4_row_bytes(D_IDX);
        for (int i = threadIdx.x; i < H_I * D_IDX; i += blockDim.x) {
            const int h = i / D_IDX, d = i % D_IDX;
            const uint8_t* row = q8 + h * mxfp4_row_bytes(D_IDX);
            const uint32_t code = (row[d >> 1] >> (4 * (d & 1))) & 0xF;
            qs[i] = e2m1_to_f32(code) * e8m0_to_f32(row[D_IDX / 2 + d / 32]);
        }
    } else {
        const TQ* qrow = reinterpret_cast<const TQ*>(qI) + bq * (int64_t)H_I * D_IDX;
        for (int i = threadIdx.x; i < H_I * D_IDX; i += blockDim.x) qs[i] = to_f32<TQ>(qrow[i]);
    }
}

template <typename TQ, int KF>
__global__ void __launch_bounds__(SIMT_TILE) index_score_simt_kernel(
    const void* __restrict__ qI, const float* __restrict__ w, const void* __restrict__ kI, int Q, int64_t N,
    int H_I, const int64_t* __restrict__ n_visible, const int32_t* __restrict__ pool, int n_pool, int block,
    float* __restrict__ scores, float* __restrict__ bmax, unsigned int* st) {
    extern __shared__ float smem[];
    float* qs = smem;                      // [H_I][128]
    float* ws = smem + H_I * D_IDX;        // [H_I]
    const int64_t bq = blockIdx.y;         // b * Q + q
    const int64_t b = bq / Q;
    load_queries<TQ>(qI, bq, H_I, qs);
    for (int i = threadIdx.x; i < H_I; i += blockDim.x) ws[i] = w[bq * H_I + i];
    __syncthreads();

    const int64_t V = n_visible[bq];
    const bool cand = pool != nullptr;
    const int64_t n_elems = cand ? (int64_t)n_pool * block : N;
    const int64_t e = (int64_t)blockIdx.x * SIMT_TILE + threadIdx.x;
    int64_t s = e;
    bool valid = e < n_elems;
    if (cand && valid) {
        int32_t pb = pool[bq * n_pool + e / block];
        s = (int64_t)pb * block + e % block;
        valid = pb >= 0 && s < V;
        if (pb >= 0 && s >= N && s < V) { csa2_flag(st, CSA2_DEVBIT_RANGE); valid = false; }
    } else if (valid) {
        valid = s < V;
    }
    float score = -INFINITY;
    if (valid) {
        float k[D_IDX];
        load_key_row<KF>(kI, b * N + s, k);
        float acc = 0.0f;
        for (int h = 0; h < H_I; ++h) {
            const float4* qh = reinterpret_cast<const float4*>(qs + h * D_IDX);
            float dot = 0.0f;
#pragma unroll
            for (int i = 0; i < D_IDX / 4; ++i) {
                float4 qv = qh[i];
                dot = fmaf(qv.x, k[4 * i], dot);
                dot = fmaf(qv.y, k[4 * i + 1], dot);
                dot = fmaf(qv.z, k[4 * i + 2], dot);
                dot = fmaf(qv.w, k[4 * i + 3], dot);
            }
            acc = fmaf(ws[h], fmaxf(dot, 0.0f), acc);
        }
        score = acc;
    }
    if (e < n_elems && scores) scores[bq * n_elems + e] = score;
    if (!cand && bmax) {
        // block max over `block` consecutive lanes (block is a power of two <= 32)
        float v = score;
        for (int o = 1; o < block; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        const int64_t nb = (N + block - 1) / block;
        if ((e % block) == 0 && e / block < nb) bmax[bq * nb + e / block] = v;
    }
}

template <typename TQ, int KF>
void launch_simt(const void* qI, const float* w, const void* kI, int B, int Q, int64_t N, int H_I,
                 const int64_t* nv, const int32_t* pool, int n_pool, int block, float* scores, float* bmax,
                 unsigned int* st, cudaStream_t s) {
    const int64_t n_elems = pool ? (int64_t)n_pool * block : N;
    dim3 grid((unsigned)((n_elems + SIMT_TILE - 1) / SIMT_TILE), (unsigned)(B * Q));
    size_t sm = (size_t)(H_I * D_IDX + H_I) * sizeof(float);
    if (sm > 48 * 1024)
        cudaFuncSetAttribute(index_score_simt_kernel<TQ, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    index_score_simt_kernel<TQ, KF><<<grid, SIMT_TILE, sm, s>>>(qI, w, kI, Q, N, H_I, nv, pool,
                                                                 n_pool, block, scores, bmax, st);
}

// Entries visible to each query: entry j needs t >= m(j+1), so floor(t/m) of them
// (a negative position sees none).
__global__ void visible_kernel(const int64_t* q_pos, int64_t rows, int m, int64_t* nv) {
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = q_pos[i];
        nv[i] = t >= 0 ? t / m : 0;
    }
    pdl_trigger();
}

}  // namespace

extern "C" csa2_status csa2_visible_entries(csa2_ctx* ctx, const int64_t* q_pos, int64_t rows, int m,
                                            int64_t* n_visible, void* stream) {
    if (!ctx || rows < 0 || m < 1) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (!q_pos || !n_visible) return CSA2_ERR_INVALID_ARG;
    const int64_t blocks = std::min<int64_t>((rows + 255) / 256, 4 * (int64_t)ctx->num_sms);
    return launch_pdl(visible_kernel, dim3((unsigned)blocks), dim3(256), 0, as_stream(stream), q_pos, rows, m,
                      n_visible);
}

extern "C" csa2_status csa2_index_score_mxq(csa2_ctx* ctx, const void* q_bf16, const float* w, const void* k_idx,
                                            int B, int Q, int64_t N, int H_I, int d_I, const int64_t* n_visible,
                                            int block, float* scores, float* block_max, uint32_t* block_hist,
                                            uint8_t* q_mx_out, void* stream) {
    if (!ctx || B < 0 || Q < 0 || N < 0 || H_I < 1) return CSA2_ERR_INVALID_ARG;
    if (d_I != D_IDX || H_I != 64 || block != 8 || (N % 8) != 0) return CSA2_ERR_UNSUPPORTED;
    if (block_hist && !block_max) return CSA2_ERR_INVALID_ARG;
    if ((int64_t)B * Q > 65535) return CSA2_ERR_UNSUPPORTED;
    if (B == 0 || Q == 0 || N == 0) return CSA2_OK;
    if (!q_bf16 || !w || !n_visible || !k_idx) return CSA2_ERR_INVALID_ARG;
    if (!aligned(q_bf16, 16) || !aligned(k_idx, 16) || (block_hist && !aligned(block_hist, 16)))
        return CSA2_ERR_INVALID_ARG;
    if (q_mx_out && !aligned(q_mx_out, 4)) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (block_hist) {
        const csa2_status z = block_hist_zero(block_hist, (int64_t)B * Q, s);
        if (z != CSA2_OK) return z;
    }
    return index_score_fp4_dispatch(ctx, nullptr, w, k_idx, B, Q, N, H_I, n_visible, nullptr, 0, block, scores,
                                    block_max, block_hist, s, q_bf16, q_mx_out);
}

extern "C" csa2_status csa2_index_score(csa2_ctx* ctx, const void* q_idx, csa2_dtype q_dt, const float* w,
                                        const void* k_idx, csa2_dtype k_dt, int B, int Q, int64_t N, int H_I,
                                        int d_I, const int64_t* n_visible, const int32_t* pool_blocks,
                                        int n_pool, int block, float* scores, float* block_max,
                                        uint32_t* block_hist, void* stream) {
    if (!ctx || B < 0 || Q < 0 || N < 0 || H_I < 1 || H_I > 128) return CSA2_ERR_INVALID_ARG;
    if (d_I != D_IDX) return CSA2_ERR_UNSUPPORTED;
    if (block < 1 || block > 32 || (block & (block - 1))) return CSA2_ERR_INVALID_ARG;
    if (pool_blocks && (block_max || !scores || n_pool < 0)) return CSA2_ERR_INVALID_ARG;
    if (block_hist && (pool_blocks || !block_max)) return CSA2_ERR_INVALID_ARG;
    if (q_dt != CSA2_F32 && q_dt != CSA2_BF16 && q_dt != CSA2_MXFP4_E8M0x32) return CSA2_ERR_UNSUPPORTED;
    if (k_dt != CSA2_F32 && k_dt != CSA2_BF16 && k_dt != CSA2_MXFP4_E8M0x32) return CSA2_ERR_UNSUPPORTED;
    if ((int64_t)B * Q > 65535) return CSA2_ERR_UNSUPPORTED;
    if (B == 0 || Q == 0) return CSA2_OK;
    if (!q_idx || !w || !n_visible || (N > 0 && !k_idx)) return CSA2_ERR_INVALID_ARG;
    if (!aligned(q_idx, 16) || !aligned(k_idx, 16)) return CSA2_ERR_INVALID_ARG;
    const int64_t n_elems = pool_blocks ? (int64_t)n_pool * block : N;
    if (n_elems == 0) return CSA2_OK;
    if (block_hist && !aligned(block_hist, 16)) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    const int64_t rows = (int64_t)B * Q;
    if (block_hist) {
        const csa2_status z = block_hist_zero(block_hist, rows, s);
        if (z != CSA2_OK) return z;
    }
    // the histogram of the block maxima: built by the FP4 scan itself, else counted
    // from the written maxima once the scan is done
    auto hist_after = [&](csa2_status r) -> csa2_status {
        if (r != CSA2_OK || !block_hist) return r;
        return block_hist_from_max(block_max, rows, (N + block - 1) / block, n_visible, block, block_hist, s);
    };

    // FP4 tensor-core scan for MXFP4 queries over MXFP4 keys; the kind::f16 scan for
    // bf16 queries over bf16 or MXFP4 keys.
    if (q_dt == CSA2_MXFP4_E8M0x32 && k_dt == CSA2_MXFP4_E8M0x32) {
        csa2_status r = index_score_fp4_dispatch(ctx, q_idx, w, k_idx, B, Q, N, H_I, n_visible, pool_blocks, n_pool,
                                                 block, scores, block_max, block_hist, s);
        if (r != CSA2_ERR_UNSUPPORTED) return r;
    }
    if (q_dt == CSA2_BF16 && k_dt != CSA2_F32) {
        csa2_status r = index_score_tc_dispatch(ctx, q_idx, w, k_idx, k_dt, B, Q, N, H_I, n_visible,
                                                pool_blocks, n_pool, block, scores, block_max, s);
        if (r != CSA2_ERR_UNSUPPORTED) return hist_after(r);
    }
#define CSA2_IS_LAUNCH(TQ, KF)                                                                            \
    launch_simt<TQ, KF>(q_idx, w, k_idx, B, Q, N, H_I, n_visible, pool_blocks, n_pool, block, scores,       \
                        block_max, ctx->status, s)
    if (q_dt == CSA2_MXFP4_E8M0x32) {
        if (k_dt == CSA2_F32) CSA2_IS_LAUNCH(QMx, K_F32);
        else if (k_dt == CSA2_BF16) CSA2_IS_LAUNCH(QMx, K_BF16);
        else CSA2_IS_LAUNCH(QMx, K_MX);
    } else if (q_dt == CSA2_F32) {
        if (k_dt == CSA2_F32) CSA2_IS_LAUNCH(float, K_F32);
        else if (k_dt == CSA2_BF16) CSA2_IS_LAUNCH(float, K_BF16);
        else CSA2_IS_LAUNCH(float, K_MX);
    } else {
        if (k_dt == CSA2_F32) CSA2_IS_LAUNCH(__nv_bfloat16, K_F32);
        else if (k_dt == CSA2_BF16) CSA2_IS_LAUNCH(__nv_bfloat16, K_BF16);
        else CSA2_IS_LAUNCH(__nv_bfloat16, K_MX);
    }
#undef CSA2_IS_LAUNCH
    return hist_after(csa2_launch_status());
}
