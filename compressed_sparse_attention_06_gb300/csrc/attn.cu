// Shared-KV MQA over the selected compressed entries plus the sliding window
// (DSA-to-CSA/HCA page eqs. (18)-(19) and (27), «因果边界与短滑窗»; CSA2 page
// «保留了 CSA 的骨架»): the same (RMS-normalised) row is key and value for every
// head; the query is RMSNorm'd and rotated by RoPE_t on its last 64 dims; the
// output is rotated back by RoPE_-t; the sink adds e^{z'_h} to the denominator only.
//
// CUDA-core kernel: a CTA per (query, group of 8 heads), one warp per head.  Key
// slots (the k selected ids, then the window positions) are processed in chunks of
// 32 rows staged in shared memory as f32 (FP4 rows are dequantised on the way in);
// each lane owns channels lane + 32 i of its head's query and accumulator, logits
// are warp reductions, and the softmax is online (running max, running sum).
#include "csa2_internal.cuh"

namespace {

constexpr int ATT_HG = 8;            // heads per CTA (one warp each)
constexpr int ATT_THREADS = 32 * ATT_HG;
constexpr int ATT_KC = 32;           // key rows per chunk
constexpr int ATT_C = 512;           // head dim this kernel is built for
constexpr int ATT_PER_LANE = ATT_C / 32;

enum KvKind { KV_F32 = 0, KV_BF16 = 1, KV_FP4 = 2 };

// Load 16 channels [16*lane, 16*lane+16) of a row into f32.
template <int KIND>
__device__ __forceinline__ void load_row16(const void* base, int64_t row, int lane, float (&v)[16]) {
    if (KIND == KV_F32) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + row * ATT_C + 16 * lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 u = p[i];
            v[4 * i] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
        }
    } else if (KIND == KV_BF16) {
        const uint4* p = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + row * ATT_C + 16 * lane);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint4 u = p[i];
            uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        }
    } else {
        const uint8_t* r = reinterpret_cast<const uint8_t*>(base) + row * fp4_row_bytes(ATT_C);
        uint2 codes = *reinterpret_cast<const uint2*>(r + 8 * lane);
        float s = e4m3_to_f32(r[ATT_C / 2 + lane]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = e2m1_to_f32((codes.x >> (4 * j)) & 0xF) * s;
            v[8 + j] = e2m1_to_f32((codes.y >> (4 * j)) & 0xF) * s;
        }
    }
}

template <typename TQ, int KVK, typename TS, typename TO>
__global__ void __launch_bounds__(ATT_THREADS) sparse_attn_simt_kernel(
    const TQ* __restrict__ q, const void* __restrict__ kv, int64_t N, const int32_t* __restrict__ idx, int k,
    const TS* __restrict__ swa, int64_t swa_cap, int64_t swa_pos0, int window, const int64_t* __restrict__ q_pos,
    const float* __restrict__ sink, int Q, int H, float rope_base, unsigned flags, TO* __restrict__ out,
    float* __restrict__ lse, unsigned int* st) {
    extern __shared__ float smem[];
    float* xs = smem;                                  // [ATT_KC][ATT_C]
    float* rinv = xs + ATT_KC * ATT_C;                 // [ATT_KC]
    int* slot_ref = reinterpret_cast<int*>(rinv + ATT_KC);   // [ATT_KC] >=0 entry id, <-1 window, -1 none

    const int64_t bq = blockIdx.x;
    const int64_t b = bq / Q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * ATT_HG + warp;
    const bool head_ok = h < H;
    const int64_t t = q_pos[bq];
    const float inv_sqrt_c = 1.0f / sqrtf((float)ATT_C);

    // ---- query: RMSNorm, RoPE_t; lane owns channels lane + 32 i ----
    float qv[ATT_PER_LANE];
    float acc[ATT_PER_LANE];
#pragma unroll
    for (int i = 0; i < ATT_PER_LANE; ++i) {
        qv[i] = head_ok ? to_f32<TQ>(q[(bq * H + h) * (int64_t)ATT_C + lane + 32 * i]) : 0.0f;
        acc[i] = 0.0f;
    }
    if (flags & CSA2_QNORM) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) ss = fmaf(qv[i], qv[i], ss);
        ss = warp_sum(ss);
        float r = 1.0f / sqrtf(ss / (float)ATT_C + 1e-6f);
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) qv[i] *= r;
    }
    // RoPE pair (448+2j, 449+2j) = (even lane, odd lane) of chunks i = 14, 15
    float rc[2], rs[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        int ch = lane + 32 * (14 + i);
        int j = (ch - (ATT_C - 64)) >> 1;
        rope_cos_sin(t, j, rope_base, rc[i], rs[i]);
    }
    if (flags & CSA2_ROPE) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float x = qv[14 + i];
            float p = __shfl_xor_sync(0xffffffffu, x, 1);
            qv[14 + i] = (lane & 1) ? fmaf(p, rs[i], x * rc[i]) : fmaf(-p, rs[i], x * rc[i]);
        }
    }

    float m_run = -INFINITY, l_run = 0.0f;
    const int nw = (int)max((int64_t)0, min((int64_t)window, t + 1));   // window rows present (positions >= 0)
    const int n_slots = k + nw;
    for (int c0 = 0; c0 < n_slots; c0 += ATT_KC) {
        // ---- stage the chunk: warp w loads rows w, w+8, w+16, w+24 ----
        for (int r = warp; r < ATT_KC; r += ATT_HG) {
            const int sl = c0 + r;
            int ref = -1;
            bool from_window = false;
            int64_t row = 0;
            if (sl < k) {
                int32_t id = idx[bq * k + sl];
                if (id >= 0) {
                    if (id < N) { ref = id; row = b * N + id; }
                    else if (lane == 0) csa2_flag(st, CSA2_DEVBIT_RANGE);
                }
            } else if (sl < n_slots) {
                int64_t p = t - nw + 1 + (sl - k);
                int64_t slot = ((p - swa_pos0) % swa_cap + swa_cap) % swa_cap;
                ref = -2;
                from_window = true;
                row = b * swa_cap + slot;
            }
            float v[16];
            if (ref != -1) {
                if (from_window) {
                    if (sizeof(TS) == 4) load_row16<KV_F32>(swa, row, lane, v);
                    else load_row16<KV_BF16>(swa, row, lane, v);
                } else {
                    load_row16<KVK>(kv, row, lane, v);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.0f;
            }
            float ss = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) ss = fmaf(v[j], v[j], ss);
            ss = warp_sum(ss);
            float4* dst = reinterpret_cast<float4*>(xs + r * ATT_C + 16 * lane);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            if (lane == 0) {
                rinv[r] = (flags & CSA2_KVNORM) ? 1.0f / sqrtf(ss / (float)ATT_C + 1e-6f) : 1.0f;
                slot_ref[r] = ref;
            }
        }
        __syncthreads();
        // ---- logits: lane j ends up holding key j's logit ----
        float z_mine = -INFINITY;
        const int n_here = min(ATT_KC, n_slots - c0);
        for (int j = 0; j < n_here; ++j) {
            const float* xr = xs + j * ATT_C;
            float d = 0.0f;
#pragma unroll
            for (int i = 0; i < ATT_PER_LANE; ++i) d = fmaf(qv[i], xr[lane + 32 * i], d);
            d = warp_sum(d);
            if (lane == j && slot_ref[j] != -1) z_mine = d * rinv[j] * inv_sqrt_c;
        }
        // ---- online softmax update ----
        float cmax = warp_max(z_mine);
        float m_new = fmaxf(m_run, cmax);
        float scale = (m_new == -INFINITY) ? 1.0f : expf(m_run - m_new);
        float p_mine = (z_mine == -INFINITY) ? 0.0f : expf(z_mine - m_new);
        l_run = l_run * scale + warp_sum(p_mine);
        m_run = m_new;
        float pr = p_mine * rinv[lane];
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) acc[i] *= scale;
        for (int j = 0; j < n_here; ++j) {
            float pj = __shfl_sync(0xffffffffu, pr, j);
            if (pj == 0.0f) continue;
            const float* xr = xs + j * ATT_C;
#pragma unroll
            for (int i = 0; i < ATT_PER_LANE; ++i) acc[i] = fmaf(pj, xr[lane + 32 * i], acc[i]);
        }
        __syncthreads();
    }
    if (!head_ok) return;
    // ---- sink, normalisation, inverse RoPE, store ----
    float zs = sink ? sink[h] : -INFINITY;
    float m_fin = fmaxf(m_run, zs);
    float denom, a_scale;
    if (m_fin == -INFINITY) {
        denom = 0.0f;
        a_scale = 0.0f;
    } else {
        float e_run = (m_run == -INFINITY) ? 0.0f : expf(m_run - m_fin);
        denom = l_run * e_run + ((zs == -INFINITY) ? 0.0f : expf(zs - m_fin));
        a_scale = denom > 0.0f ? e_run / denom : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < ATT_PER_LANE; ++i) acc[i] *= a_scale;
    if (flags & CSA2_ROPE) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float x = acc[14 + i];
            float p = __shfl_xor_sync(0xffffffffu, x, 1);
            // rotation by -t: (x0 c + x1 s, -x0 s + x1 c)
            acc[14 + i] = (lane & 1) ? fmaf(-p, rs[i], x * rc[i]) : fmaf(p, rs[i], x * rc[i]);
        }
    }
    TO* o = out + (bq * H + h) * (int64_t)ATT_C;
#pragma unroll
    for (int i = 0; i < ATT_PER_LANE; ++i) o[lane + 32 * i] = from_f32<TO>(acc[i]);
    if (lse && lane == 0) lse[bq * H + h] = (denom > 0.0f) ? m_fin + logf(denom) : -INFINITY;
}

template <typename TQ, int KVK, typename TS, typename TO>
csa2_status launch_attn(const void* q, const void* kv, int64_t N, const int32_t* idx, int k, const void* swa,
                        int64_t swa_cap, int64_t swa_pos0, int window, const int64_t* q_pos, const float* sink,
                        int B, int Q, int H, float base, unsigned flags, void* out, float* lse, unsigned int* st,
                        cudaStream_t s) {
    auto kern = sparse_attn_simt_kernel<TQ, KVK, TS, TO>;
    size_t sm = (size_t)ATT_KC * ATT_C * sizeof(float) + ATT_KC * sizeof(float) + ATT_KC * sizeof(int);
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess)
            return CSA2_ERR_CUDA;
        attr_set = true;
    }
    dim3 grid((unsigned)(B * Q), (unsigned)((H + ATT_HG - 1) / ATT_HG));
    kern<<<grid, ATT_THREADS, sm, s>>>((const TQ*)q, kv, N, idx, k, (const TS*)swa, swa_cap, swa_pos0, window,
                                       q_pos, sink, Q, H, base, flags, (TO*)out, lse, st);
    return csa2_launch_status();
}

template <typename TQ, int KVK, typename TS>
csa2_status dispatch_out(csa2_dtype out_dt, const void* q, const void* kv, int64_t N, const int32_t* idx, int k,
                         const void* swa, int64_t cap, int64_t p0, int window, const int64_t* q_pos,
                         const float* sink, int B, int Q, int H, float base, unsigned flags, void* out, float* lse,
                         unsigned int* st, cudaStream_t s) {
    if (out_dt == CSA2_F32)
        return launch_attn<TQ, KVK, TS, float>(q, kv, N, idx, k, swa, cap, p0, window, q_pos, sink, B, Q, H, base,
                                               flags, out, lse, st, s);
    return launch_attn<TQ, KVK, TS, __nv_bfloat16>(q, kv, N, idx, k, swa, cap, p0, window, q_pos, sink, B, Q, H,
                                                   base, flags, out, lse, st, s);
}

template <typename TQ, int KVK>
csa2_status dispatch_swa(csa2_dtype swa_dt, csa2_dtype out_dt, const void* q, const void* kv, int64_t N,
                         const int32_t* idx, int k, const void* swa, int64_t cap, int64_t p0, int window,
                         const int64_t* q_pos, const float* sink, int B, int Q, int H, float base, unsigned flags,
                         void* out, float* lse, unsigned int* st, cudaStream_t s) {
    if (swa_dt == CSA2_F32)
        return dispatch_out<TQ, KVK, float>(out_dt, q, kv, N, idx, k, swa, cap, p0, window, q_pos, sink, B, Q, H,
                                            base, flags, out, lse, st, s);
    return dispatch_out<TQ, KVK, __nv_bfloat16>(out_dt, q, kv, N, idx, k, swa, cap, p0, window, q_pos, sink, B, Q,
                                                H, base, flags, out, lse, st, s);
}

}  // namespace

extern "C" csa2_status csa2_sparse_attn(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const void* kv,
                                        csa2_dtype kv_dt, int64_t N, const int32_t* idx, int k, const void* swa,
                                        csa2_dtype swa_dt, int64_t swa_cap, int64_t swa_pos0, int window,
                                        const int64_t* q_pos, const float* sink, int B, int Q, int H, int c,
                                        float rope_base, unsigned flags, void* out, csa2_dtype out_dt, float* lse,
                                        void* stream) {
    if (!ctx || B < 0 || Q < 0 || N < 0 || k < 0 || k > 2048 || window < 0 || window > 1024) return CSA2_ERR_INVALID_ARG;
    if (H < 1 || H > 128) return CSA2_ERR_INVALID_ARG;
    if (c != ATT_C) return CSA2_ERR_UNSUPPORTED;
    if (flags & ~(CSA2_QNORM | CSA2_KVNORM | CSA2_ROPE)) return CSA2_ERR_INVALID_ARG;
    if (q_dt != CSA2_F32 && q_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (kv_dt != CSA2_F32 && kv_dt != CSA2_BF16 && kv_dt != CSA2_FP4_E4M3x16) return CSA2_ERR_UNSUPPORTED;
    if (swa_dt != CSA2_F32 && swa_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (out_dt != CSA2_F32 && out_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if ((int64_t)B * Q > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED;
    if (B == 0 || Q == 0) return CSA2_OK;
    if (!q || !q_pos || !out) return CSA2_ERR_INVALID_ARG;
    if (k > 0 && (!idx || !kv)) return CSA2_ERR_INVALID_ARG;
    if (window > 0 && (!swa || swa_cap < window)) return CSA2_ERR_INVALID_ARG;
    if (window == 0) swa_cap = 1;
    if (!aligned(kv, 16) || !aligned(swa, 16) || !aligned(q, 16)) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    unsigned int* st = ctx->status;
#define CSA2_ATT(TQ, KVK)                                                                                   \
    return dispatch_swa<TQ, KVK>(swa_dt, out_dt, q, kv, N, idx, k, swa, swa_cap, swa_pos0, window, q_pos, sink, \
                                 B, Q, H, rope_base, flags, out, lse, st, s)
    if (q_dt == CSA2_F32) {
        if (kv_dt == CSA2_F32) CSA2_ATT(float, KV_F32);
        if (kv_dt == CSA2_BF16) CSA2_ATT(float, KV_BF16);
        CSA2_ATT(float, KV_FP4);
    } else {
        if (kv_dt == CSA2_F32) CSA2_ATT(__nv_bfloat16, KV_F32);
        if (kv_dt == CSA2_BF16) CSA2_ATT(__nv_bfloat16, KV_BF16);
        CSA2_ATT(__nv_bfloat16, KV_FP4);
    }
#undef CSA2_ATT
}
