// Shared-KV MQA over the selected compressed entries plus the sliding window
// (DSA-to-CSA/HCA page eqs. (18)-(19) and (27), «因果边界与短滑窗»; CSA2 page
// «保留了 CSA 的骨架»): the same (RMS-normalised) row is key and value for every
// head; the query is RMSNorm'd and rotated by RoPE_t on its last 64 dims; the
// output is rotated back by RoPE_-t; the sink adds e^{z'_h} to the denominator only.
//
// Split-key (flash-decoding) layout: a CTA per (key split, group of 8 heads,
// query), one warp per head.  The CTA stages its key slots in chunks of 32 rows in
// shared memory as f32 (FP4 rows dequantised on the way in, with each row's RMS),
// each lane owns channels lane + 32 i of its head's query and accumulator, logits
// are warp reductions, and the softmax is online.  With one split the CTA finishes
// the head (sink, normalisation, inverse RoPE); with several, each split writes its
// partial (max, sum, unnormalised output) to the caller's workspace and
// attn_combine_kernel merges them by log-sum-exp.
#include <algorithm>
#include <cstring>

#include "attn_tc.cuh"
#include "csa2_internal.cuh"

namespace {

constexpr int ATT_HG = 8;            // heads per CTA (one warp each)
constexpr int ATT_THREADS = 32 * ATT_HG;
constexpr int ATT_KC = 32;           // key rows per staged chunk
constexpr int ATT_C = 512;           // head dim this kernel is built for
constexpr int ATT_PER_LANE = ATT_C / 32;
constexpr int PART = ATTN_PART;      // floats per partial (layout in attn_tc.cuh)
constexpr int PO = ATTN_PART_O;

enum KvKind { KV_F32 = 0, KV_BF16 = 1, KV_FP4 = 2 };

// Load 16 channels [16*lane, 16*lane+16) of a row into f32 (exact for every format).
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
        const float s = e4m3_to_f32(r[ATT_C / 2 + lane]);
        float lo[8], hi[8];
        e2m1x8_to_f32(codes.x, lo);
        e2m1x8_to_f32(codes.y, hi);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = lo[j] * s;
            v[8 + j] = hi[j] * s;
        }
    }
}

struct AttnArgs {
    const void* q;
    const void* kv;
    int64_t N;
    const int32_t* idx;
    int k;
    const int64_t* dense_nv;  // dense mode (idx NULL): entries 0 .. dense_nv[bq]-1
    const void* swa;
    int64_t swa_cap, swa_pos0;
    int window;
    const int64_t* q_pos;
    const float* sink;
    int Q, H;
    int Hs;               // heads per query in out / lse (combine of a tensor-core head pass; else H)
    RopeTable rope;
    unsigned flags;
    void* out;
    float* lse;
    float* ws;            // [B*Q, H, n_split, PART] partials (n_split > 1)
    const float* rope_cs; // [B*Q, 64] RoPE cos, sin at the query position (tensor-core path), or NULL
    int n_split;
    int spl;              // key slots per split (multiple of ATT_KC)
    unsigned int* st;
};

// Rotate this warp's channels 448..511 (lanes hold lane+448 and lane+480) by +t
// (sign = 1) or -t (sign = -1); pairs are (even lane, odd lane).
template <typename TQ, int KVK, typename TS, typename TO>
__global__ void __launch_bounds__(ATT_THREADS, 2) attn_split_kernel(const AttnArgs a) {
    extern __shared__ float smem[];
    float* xs = smem;                                   // [ATT_KC][ATT_C]
    float* rinv = xs + ATT_KC * ATT_C;                  // [ATT_KC]
    int* slot_ok = reinterpret_cast<int*>(rinv + ATT_KC);   // [ATT_KC]
    float* cs = reinterpret_cast<float*>(slot_ok + ATT_KC);  // [32] RoPE cos at t
    float* sn = cs + 32;                                      // [32] RoPE sin at t

    const int split = blockIdx.x;
    const int64_t bq = blockIdx.z;
    const int64_t b = bq / a.Q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * ATT_HG + warp;
    const bool head_ok = h < a.H;
    const int64_t t = a.q_pos[bq];
    const float inv_sqrt_c = 1.0f / sqrtf((float)ATT_C);
    const TQ* q = reinterpret_cast<const TQ*>(a.q);
    if (threadIdx.x < 32) rope_cos_sin(a.rope, t, threadIdx.x, cs[threadIdx.x], sn[threadIdx.x]);
    __syncthreads();

    float qv[ATT_PER_LANE], acc[ATT_PER_LANE];
#pragma unroll
    for (int i = 0; i < ATT_PER_LANE; ++i) {
        qv[i] = head_ok ? to_f32<TQ>(q[(bq * a.H + h) * (int64_t)ATT_C + lane + 32 * i]) : 0.0f;
        acc[i] = 0.0f;
    }
    if (a.flags & CSA2_QNORM) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) ss = fmaf(qv[i], qv[i], ss);
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss / (float)ATT_C + 1e-6f);
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) qv[i] *= r;
    }
    if (a.flags & CSA2_ROPE) rope_lanes(qv, lane, cs, sn, 1.0f);

    const int nw = (int)max((int64_t)0, min((int64_t)a.window, t + 1));   // window rows (positions >= 0)
    const int kq = a.dense_nv ? (int)max((int64_t)0, min((int64_t)a.k, a.dense_nv[bq])) : a.k;
    const int n_slots = kq + nw;
    const int s_begin = split * a.spl;
    const int s_end = min(n_slots, s_begin + a.spl);
    float m_run = -INFINITY, l_run = 0.0f;
    for (int c0 = s_begin; c0 < s_end; c0 += ATT_KC) {
        // stage the chunk: warp w loads rows w, w+8, w+16, w+24
        for (int r = warp; r < ATT_KC; r += ATT_HG) {
            const int sl = c0 + r;
            int ok = 0;
            bool from_window = false;
            int64_t row = 0;
            if (sl < s_end) {
                if (sl < kq) {
                    const int32_t id = a.dense_nv ? sl : a.idx[bq * a.k + sl];
                    if (id >= 0) {
                        if (id < a.N) { ok = 1; row = b * a.N + id; }
                        else if (lane == 0) csa2_flag(a.st, CSA2_DEVBIT_RANGE);
                    }
                } else {
                    const int64_t p = t - nw + 1 + (sl - kq);
                    const int64_t slot = ((p - a.swa_pos0) % a.swa_cap + a.swa_cap) % a.swa_cap;
                    ok = 1;
                    from_window = true;
                    row = b * a.swa_cap + slot;
                }
            }
            float v[16];
            if (ok) {
                if (from_window) {
                    if (sizeof(TS) == 4) load_row16<KV_F32>(a.swa, row, lane, v);
                    else load_row16<KV_BF16>(a.swa, row, lane, v);
                } else {
                    load_row16<KVK>(a.kv, row, lane, v);
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
                rinv[r] = (a.flags & CSA2_KVNORM) ? 1.0f / sqrtf(ss / (float)ATT_C + 1e-6f) : 1.0f;
                slot_ok[r] = ok;
            }
        }
        __syncthreads();
        // logits: lane j ends up holding key j's logit
        float z_mine = -INFINITY;
        const int n_here = min(ATT_KC, s_end - c0);
        for (int j = 0; j < n_here; ++j) {
            const float* xr = xs + j * ATT_C;
            float d = 0.0f;
#pragma unroll
            for (int i = 0; i < ATT_PER_LANE; ++i) d = fmaf(qv[i], xr[lane + 32 * i], d);
            d = warp_sum(d);
            if (lane == j && slot_ok[j]) z_mine = d * rinv[j] * inv_sqrt_c;
        }
        // online softmax update
        const float cmax = warp_max(z_mine);
        const float m_new = fmaxf(m_run, cmax);
        const float scale = (m_new == -INFINITY) ? 1.0f : expf(m_run - m_new);
        const float p_mine = (z_mine == -INFINITY) ? 0.0f : expf(z_mine - m_new);
        l_run = l_run * scale + warp_sum(p_mine);
        m_run = m_new;
        const float pr = p_mine * rinv[lane];
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) acc[i] *= scale;
        for (int j = 0; j < n_here; ++j) {
            const float pj = __shfl_sync(0xffffffffu, pr, j);
            if (pj == 0.0f) continue;
            const float* xr = xs + j * ATT_C;
#pragma unroll
            for (int i = 0; i < ATT_PER_LANE; ++i) acc[i] = fmaf(pj, xr[lane + 32 * i], acc[i]);
        }
        __syncthreads();
    }
    if (!head_ok) return;
    if (a.n_split > 1) {
        float* part = a.ws + ((bq * a.H + h) * (int64_t)a.n_split + split) * PART;
        if (lane == 0) {
            part[0] = m_run;
            part[1] = l_run;
        }
#pragma unroll
        for (int i = 0; i < ATT_PER_LANE; ++i) part[PO + lane + 32 * i] = acc[i];
        return;
    }
    // single split: sink, normalisation, inverse RoPE, store
    const float zs = a.sink ? a.sink[h] : -INFINITY;
    const float m_fin = fmaxf(m_run, zs);
    float denom = 0.0f, a_scale = 0.0f;
    if (m_fin != -INFINITY) {
        const float e_run = (m_run == -INFINITY) ? 0.0f : expf(m_run - m_fin);
        denom = l_run * e_run + ((zs == -INFINITY) ? 0.0f : expf(zs - m_fin));
        a_scale = denom > 0.0f ? e_run / denom : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < ATT_PER_LANE; ++i) acc[i] *= a_scale;
    if (a.flags & CSA2_ROPE) rope_lanes(acc, lane, cs, sn, -1.0f);
    TO* o = reinterpret_cast<TO*>(a.out) + (bq * a.H + h) * (int64_t)ATT_C;
#pragma unroll
    for (int i = 0; i < ATT_PER_LANE; ++i) o[lane + 32 * i] = from_f32<TO>(acc[i]);
    if (a.lse && lane == 0) a.lse[bq * a.H + h] = (denom > 0.0f) ? m_fin + logf(denom) : -INFINITY;
}

// Merge the splits of one (query, head) per warp: the split maxima are read one per
// lane, then four splits at a time are accumulated with all their loads in flight.
template <typename TO>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a, int64_t rows) {
    __shared__ float cs_all[8][32], sn_all[8][32];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * 8 + warp;      // (bq, h)
    if (r >= rows) return;
    const int64_t bq = r / a.H;
    const int h = (int)(r % a.H);
    float* cs = cs_all[warp];
    float* sn = sn_all[warp];
    if (a.flags & CSA2_ROPE) {
        if (a.rope_cs) {
            cs[lane] = a.rope_cs[bq * 64 + lane];
            sn[lane] = a.rope_cs[bq * 64 + 32 + lane];
        } else {
            rope_cos_sin(a.rope, a.q_pos[bq], lane, cs[lane], sn[lane]);
        }
    }
    __syncwarp();
    const int ns = a.n_split;
    const int64_t ro = bq * a.Hs + h;                      // row of out / lse
    attn_combine_row<TO>(a.ws + r * (int64_t)ns * PART, ns, a.sink ? a.sink[h] : -INFINITY,
                         (a.flags & CSA2_ROPE) ? cs : nullptr, sn, reinterpret_cast<TO*>(a.out) + ro * (int64_t)ATT_C,
                         a.lse ? a.lse + ro : nullptr);
}

constexpr size_t ATT_SMEM = (size_t)ATT_KC * ATT_C * sizeof(float) + ATT_KC * sizeof(float) + ATT_KC * sizeof(int) +
                            64 * sizeof(float);

template <typename TQ, int KVK, typename TS, typename TO>
csa2_status launch_attn(AttnArgs& a, int B, int Q, cudaStream_t s) {
    auto kern = attn_split_kernel<TQ, KVK, TS, TO>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ATT_SMEM) != cudaSuccess)
            return CSA2_ERR_CUDA;
        attr_set = true;
    }
    dim3 grid((unsigned)a.n_split, (unsigned)((a.H + ATT_HG - 1) / ATT_HG), (unsigned)(B * Q));
    kern<<<grid, ATT_THREADS, ATT_SMEM, s>>>(a);
    if (a.n_split > 1) {
        const int64_t rows = (int64_t)B * Q * a.H;
        attn_combine_kernel<TO><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a, rows);
    }
    return csa2_launch_status();
}

template <typename TO>
csa2_status launch_combine(const AttnArgs& a, int B, int Q, cudaStream_t s) {
    const int64_t rows = (int64_t)B * Q * a.H;
    const csa2_status r = launch_pdl(attn_combine_kernel<TO>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, s, a, rows);
    return r != CSA2_OK ? r : csa2_launch_status();
}

template <typename TQ, int KVK, typename TS>
csa2_status dispatch_out(csa2_dtype out_dt, AttnArgs& a, int B, int Q, cudaStream_t s) {
    if (out_dt == CSA2_F32) return launch_attn<TQ, KVK, TS, float>(a, B, Q, s);
    return launch_attn<TQ, KVK, TS, __nv_bfloat16>(a, B, Q, s);
}

template <typename TQ, int KVK>
csa2_status dispatch_swa(csa2_dtype swa_dt, csa2_dtype out_dt, AttnArgs& a, int B, int Q, cudaStream_t s) {
    if (swa_dt == CSA2_F32) return dispatch_out<TQ, KVK, float>(out_dt, a, B, Q, s);
    return dispatch_out<TQ, KVK, __nv_bfloat16>(out_dt, a, B, Q, s);
}

// Number of key splits: about two waves of CTAs, at least 32 slots per split, and
// no more than the workspace holds.
int choose_splits(const csa2_ctx* ctx, int64_t groups, int n_slots_max, int64_t rows_bqh, size_t ws_bytes,
                  bool have_ws) {
    const int64_t target = 4LL * ctx->num_sms;
    int want = 1;
    if (groups < target) want = (int)((target + groups - 1) / groups);
    const int max_by_slots = (n_slots_max + ATT_KC - 1) / ATT_KC;
    want = std::min(want, std::max(1, max_by_slots));
    if (!have_ws || want <= 1) return 1;
    const int64_t fit = (int64_t)(ws_bytes / ((size_t)rows_bqh * PART * sizeof(float)));
    if (fit < 2) return 1;
    return (int)std::min<int64_t>(want, fit);
}

}  // namespace

size_t attn_simt_ws_bytes(const csa2_ctx* ctx, int B, int Q, int H, int k, int window) {
    if (!ctx || B <= 0 || Q <= 0 || H <= 0 || k < 0 || window < 0) return 0;
    const int64_t groups = (int64_t)B * Q * ((H + ATT_HG - 1) / ATT_HG);
    const int splits = choose_splits(ctx, groups, k + window, (int64_t)B * Q * H, SIZE_MAX / 2, true);
    if (splits <= 1) return 0;
    return (size_t)B * Q * H * splits * PART * sizeof(float);
}

extern "C" size_t csa2_sparse_attn_workspace_bytes(csa2_ctx* ctx, int B, int Q, int H, int k, int window, int64_t N,
                                                   int64_t swa_cap) {
    if (!ctx || B <= 0 || Q <= 0 || H <= 0 || k < 0 || window < 0 || N < 0 || swa_cap < 0) return 0;
    return std::max(attn_simt_ws_bytes(ctx, B, Q, H, k, window),
                    H > 64 ? attn_tc_ws_bytes_all_passes(ctx, B, Q, H, k, window, N, swa_cap)
                           : attn_tc_ws_bytes(ctx, B, Q, H, k, window, N, swa_cap));
}

// Sparse (idx) or dense (dense_nv: entries 0 .. dense_nv[bq]-1, at most k) attention.
static csa2_status attn_impl(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const void* kv, csa2_dtype kv_dt,
                             int64_t N, const int32_t* idx, const int64_t* dense_nv, int k, const void* swa,
                             csa2_dtype swa_dt, int64_t swa_cap, int64_t swa_pos0, int window, const int64_t* q_pos,
                             const float* sink, int B, int Q, int H, int c, float rope_base, unsigned flags, void* out,
                             csa2_dtype out_dt, float* lse, void* ws, size_t ws_bytes, void* stream) {
    if (!ctx || B < 0 || Q < 0 || N < 0 || k < 0 || window < 0 || window > 1024) return CSA2_ERR_INVALID_ARG;
    if (H < 1 || H > 128) return CSA2_ERR_INVALID_ARG;
    if (c != ATT_C) return CSA2_ERR_UNSUPPORTED;
    if (flags & ~(CSA2_QNORM | CSA2_KVNORM | CSA2_ROPE | CSA2_ATTN_PREPARED)) return CSA2_ERR_INVALID_ARG;
    // a prepared query image is used only by a single tensor-core pass (<= 64 heads);
    // otherwise the call prepares its own
    if (H > 64) flags &= ~CSA2_ATTN_PREPARED;
    if (q_dt != CSA2_F32 && q_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (kv_dt != CSA2_F32 && kv_dt != CSA2_BF16 && kv_dt != CSA2_FP4_E4M3x16) return CSA2_ERR_UNSUPPORTED;
    if (swa_dt != CSA2_F32 && swa_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (out_dt != CSA2_F32 && out_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if ((int64_t)B * Q > 65535) return CSA2_ERR_UNSUPPORTED;     // one grid.z slice per query
    if (B == 0 || Q == 0) return CSA2_OK;
    if (!q || !q_pos || !out) return CSA2_ERR_INVALID_ARG;
    if (k > 0 && ((!idx && !dense_nv) || !kv)) return CSA2_ERR_INVALID_ARG;
    if (window > 0 && (!swa || swa_cap < window)) return CSA2_ERR_INVALID_ARG;
    if (window == 0) swa_cap = 1;
    if (!aligned(kv, 16) || !aligned(swa, 16) || !aligned(q, 16) || !aligned(ws, 16)) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    // tensor-core path: bf16 query and window, bf16 or FP4 rows, both RMSNorms; heads
    // in passes of at most 64 (each pass gathers the rows once)
    AttnTcCall tc;
    tc.q = q;
    tc.q_dt = q_dt;
    tc.kv = kv;
    tc.kv_dt = kv_dt;
    tc.N = N;
    tc.idx = idx;
    tc.k = k;
    tc.dense_nv = dense_nv;
    tc.swa = swa;
    tc.swa_dt = swa_dt;
    tc.swa_cap = swa_cap;
    tc.swa_pos0 = swa_pos0;
    tc.window = window;
    tc.q_pos = q_pos;
    tc.sink = sink;
    tc.B = B;
    tc.Q = Q;
    tc.H = std::min(H, 64);
    tc.Hs = H;
    tc.rope = make_rope_table(rope_base);
    tc.flags = flags;
    tc.out = out;
    tc.out_dt = out_dt;
    tc.lse = lse;
    const size_t qsz = q_dt == CSA2_F32 ? 4 : 2, osz = out_dt == CSA2_F32 ? 4 : 2;
    // more than 64 heads: every pass in one launch when the workspace holds them all
    // (the passes' items then share one wave of CTAs); the per-pass partials merge in
    // the kernel (cluster) or in one combine launch per pass
    const int n_pass = (H + 63) / 64;
    if (attn_tc_applies(tc) && ws && n_pass > 1 &&
        ws_bytes >= attn_tc_ws_bytes_all_passes(ctx, B, Q, H, k, window, 0, 0)) {
        AttnTcCall p = tc;
        p.n_pass = n_pass;
        int ns = 1;
        const csa2_status st = attn_tc_run(ctx, p, ws, ws_bytes, s, &ns);
        if (st != CSA2_OK || ns <= 1) return st;
        const int64_t n_bq = (int64_t)B * Q;
        for (int h0 = 0; h0 < H; h0 += 64) {
            AttnArgs c;
            memset(&c, 0, sizeof(c));
            c.q_pos = q_pos;
            c.sink = sink ? sink + h0 : nullptr;
            c.Q = Q;
            c.H = std::min(64, H - h0);
            c.Hs = H;
            c.rope = tc.rope;
            c.flags = flags;
            c.out = reinterpret_cast<uint8_t*>(out) + (size_t)h0 * ATT_C * osz;
            c.lse = lse ? lse + h0 : nullptr;
            c.ws = reinterpret_cast<float*>(ws) + (size_t)h0 * n_bq * ns * PART;
            c.rope_cs = attn_tc_rope_table(ctx, p, ws);
            c.n_split = ns;
            c.st = ctx->status;
            const csa2_status sc =
                out_dt == CSA2_F32 ? launch_combine<float>(c, B, Q, s) : launch_combine<__nv_bfloat16>(c, B, Q, s);
            if (sc != CSA2_OK) return sc;
        }
        return CSA2_OK;
    }
    if (attn_tc_applies(tc) && ws && ws_bytes >= attn_tc_ws_bytes(ctx, B, Q, tc.H, k, window, 0, 0)) {
        for (int h0 = 0; h0 < H; h0 += 64) {
            AttnTcCall p = tc;
            p.H = std::min(64, H - h0);
            p.q = reinterpret_cast<const uint8_t*>(q) + (size_t)h0 * ATT_C * qsz;
            p.out = reinterpret_cast<uint8_t*>(out) + (size_t)h0 * ATT_C * osz;
            p.lse = lse ? lse + h0 : nullptr;
            p.sink = sink ? sink + h0 : nullptr;
            int ns = 1;
            const csa2_status st = attn_tc_run(ctx, p, ws, ws_bytes, s, &ns);
            if (st != CSA2_OK) return st;
            if (ns <= 1) continue;
            AttnArgs c;
            memset(&c, 0, sizeof(c));
            c.q_pos = q_pos;
            c.sink = p.sink;
            c.Q = Q;
            c.H = p.H;
            c.Hs = H;
            c.rope = tc.rope;
            c.flags = flags;
            c.out = p.out;
            c.lse = p.lse;
            c.ws = reinterpret_cast<float*>(ws);
            c.rope_cs = attn_tc_rope_table(ctx, p, ws);
            c.n_split = ns;
            c.st = ctx->status;
            const csa2_status sc =
                out_dt == CSA2_F32 ? launch_combine<float>(c, B, Q, s) : launch_combine<__nv_bfloat16>(c, B, Q, s);
            if (sc != CSA2_OK) return sc;
        }
        return CSA2_OK;
    }
    AttnArgs a;
    a.q = q;
    a.kv = kv;
    a.N = N;
    a.idx = idx;
    a.k = k;
    a.dense_nv = dense_nv;
    a.swa = swa;
    a.swa_cap = swa_cap;
    a.swa_pos0 = swa_pos0;
    a.window = window;
    a.q_pos = q_pos;
    a.sink = sink;
    a.Q = Q;
    a.H = H;
    a.Hs = H;
    a.rope = make_rope_table(rope_base);
    a.flags = flags & ~CSA2_ATTN_PREPARED;
    a.out = out;
    a.lse = lse;
    a.ws = reinterpret_cast<float*>(ws);
    a.rope_cs = nullptr;
    a.st = ctx->status;
    const int64_t groups = (int64_t)B * Q * ((H + ATT_HG - 1) / ATT_HG);
    const int n_slots_max = k + window;
    a.n_split = choose_splits(ctx, groups, n_slots_max, (int64_t)B * Q * H, ws_bytes, ws != nullptr);
    a.spl = ((n_slots_max + a.n_split - 1) / a.n_split + ATT_KC - 1) / ATT_KC * ATT_KC;
    if (a.spl == 0) a.spl = ATT_KC;
    a.n_split = std::max(1, (n_slots_max + a.spl - 1) / a.spl);
#define CSA2_ATT(TQ, KVK) return dispatch_swa<TQ, KVK>(swa_dt, out_dt, a, B, Q, s)
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

extern "C" csa2_status csa2_sparse_attn(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const void* kv,
                                        csa2_dtype kv_dt, int64_t N, const int32_t* idx, int k, const void* swa,
                                        csa2_dtype swa_dt, int64_t swa_cap, int64_t swa_pos0, int window,
                                        const int64_t* q_pos, const float* sink, int B, int Q, int H, int c,
                                        float rope_base, unsigned flags, void* out, csa2_dtype out_dt, float* lse,
                                        void* ws, size_t ws_bytes, void* stream) {
    if (k > 2048) return CSA2_ERR_INVALID_ARG;
    return attn_impl(ctx, q, q_dt, kv, kv_dt, N, idx, nullptr, k, swa, swa_dt, swa_cap, swa_pos0, window, q_pos, sink,
                     B, Q, H, c, rope_base, flags, out, out_dt, lse, ws, ws_bytes, stream);
}

extern "C" csa2_status csa2_dense_attn(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const void* kv,
                                       csa2_dtype kv_dt, int64_t N, const int64_t* n_visible, int k_max,
                                       const void* swa, csa2_dtype swa_dt, int64_t swa_cap, int64_t swa_pos0,
                                       int window, const int64_t* q_pos, const float* sink, int B, int Q, int H,
                                       int c, float rope_base, unsigned flags, void* out, csa2_dtype out_dt,
                                       float* lse, void* ws, size_t ws_bytes, void* stream) {
    if (k_max < 0 || k_max > (1 << 22) || (k_max > 0 && !n_visible)) return CSA2_ERR_INVALID_ARG;
    return attn_impl(ctx, q, q_dt, kv, kv_dt, N, nullptr, n_visible, k_max, swa, swa_dt, swa_cap, swa_pos0, window,
                     q_pos, sink, B, Q, H, c, rope_base, flags, out, out_dt, lse, ws, ws_bytes, stream);
}

extern "C" csa2_status csa2_attn_prepare(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const int64_t* q_pos, int B,
                                         int Q, int H, int c, int k, int window, int64_t N, int64_t swa_cap,
                                         float rope_base, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
    if (!ctx || B < 0 || Q < 0 || k < 0 || window < 0 || window > 1024 || H < 1 || H > 64) return CSA2_ERR_INVALID_ARG;
    if (c != ATT_C) return CSA2_ERR_UNSUPPORTED;
    if (flags & ~(CSA2_QNORM | CSA2_KVNORM | CSA2_ROPE)) return CSA2_ERR_INVALID_ARG;
    if (q_dt != CSA2_F32 && q_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if ((int64_t)B * Q > 65535) return CSA2_ERR_UNSUPPORTED;
    if (B == 0 || Q == 0) return CSA2_OK;
    if (!q || !q_pos || !aligned(q, 16) || !aligned(ws, 16)) return CSA2_ERR_INVALID_ARG;
    if (window == 0) swa_cap = 1;
    AttnTcCall tc;
    memset(&tc, 0, sizeof(tc));
    tc.n_pass = 1;
    tc.q = q;
    tc.q_dt = q_dt;
    tc.N = N;
    tc.k = k;
    tc.window = window;
    tc.swa_cap = swa_cap;
    tc.q_pos = q_pos;
    tc.B = B;
    tc.Q = Q;
    tc.H = H;
    tc.Hs = H;
    tc.rope = make_rope_table(rope_base);
    tc.flags = flags;
    return attn_tc_prepare(ctx, tc, ws, ws_bytes, as_stream(stream));
}
