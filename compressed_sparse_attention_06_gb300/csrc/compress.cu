// Gated token compressor with its write epilogue.
//
// Non-overlapping form: Attention-evolution page §4.1 and DSA-to-CSA/HCA page
// eqs. (22)-(23).  Overlapping form: DSA-to-CSA/HCA page eqs. (11)-(12), block 0
// without history (Z^b = -inf, C^b = 0) unless the previous block's state is
// carried (Attention-evolution page §3.3).  Epilogue: RMSNorm (kv_norm) -> RoPE on
// the last 64 channels at position pos0 + m*i -> f32 / bf16 / FP4 store.
//
// One CTA per compressed entry, c/4 threads, each owning 4 adjacent channels, so
// loads are coalesced float4 / 8-byte vectors, a 16-channel FP4 group is 4 adjacent
// lanes and a 32-channel MXFP4 group 8.
//
// Decode step (compress_step_kernel): the compressor state of the Attention-evolution
// page §3.3 -- the unfinished block's projections and gate logits, and the previous
// block's overlap half -- lives in a caller-owned buffer; each step stores the new
// token's rows into its slot, and the token that completes a block emits the block's
// entry into the cache (a compressed entry exists only once its block is complete,
// DSA-to-CSA/HCA page «因果边界与短滑窗»), then keeps the block's overlap half for the
// next one.
#include <algorithm>

#include "csa2_internal.cuh"

namespace {

template <typename T> __device__ __forceinline__ float4 load4(const T* p);
template <> __device__ __forceinline__ float4 load4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xFFFF0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xFFFF0000u);
    return r;
}

__device__ __forceinline__ float4 load4_bias(const float* b, int64_t off) {
    return b ? *reinterpret_cast<const float4*>(b + off) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ float f4get(const float4& v, int k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

enum OutKind { OUT_F32 = 0, OUT_BF16 = 1, OUT_FP4 = 2, OUT_MX = 3 };

constexpr int CMP_MAX_THREADS = 1024;

// Row groups of one entry's CTA: a long block (HCA's m' = 128) would leave each
// thread a serial walk over m rows, so blocks of 16 rows or more are split into up to
// m/8 groups of c/4 threads (at most CMP_MAX_THREADS threads); short blocks (CSA's
// m = 4) keep one group.
int compress_row_groups(int m, int c) {
    if (m < 16) return 1;
    return std::max(1, std::min(m / 8, CMP_MAX_THREADS / (c / 4)));
}

// Dynamic shared memory of an entry's CTA: the groups' exchange buffer, none for one group.
size_t compress_smem(int m, int c) {
    const int R = compress_row_groups(m, c);
    return R > 1 ? (size_t)2 * R * (c / 4) * sizeof(float4) : 0;
}

template <typename T>
__device__ __forceinline__ void copy4(T* dst, const T* src) {
    if (sizeof(T) == 4)
        *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(src);
    else
        *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
}

// One compressed entry; this thread's channels ch .. ch+3.  blockDim.x = R * c/4: R
// row groups (R = compress_row_groups(m, c)), group rg taking rows rg, rg+R, ... of the
// block (and of the history).  The softmax over the block's m rows (and the m history
// rows, if any) per channel, the weighted sum, then RMSNorm -> RoPE at `pos` -> store
// as row `orow` of out.  The groups share the per-channel maximum, so every row's
// weight exp(z + b - max) is the same for any R; their partial sums are added in group
// order.  Every kernel that writes entries takes its R from compress_row_groups, so an
// entry is the same bits whichever kernel (whole sequence, packed samples, decode
// step) produced it.
template <typename T, int OUT, int MAXT>
__device__ __forceinline__ void compress_entry(const T* cur_c, const T* cur_z, const T* hc, const T* hz,
                                               const float* ba, const float* bb, int c, int m, int64_t pos,
                                               const RopeTable& rope, unsigned flags, void* out, int64_t orow) {
    const int tid = threadIdx.x;
    const int cq = c >> 2;
    const int R = MAXT > 256 ? (int)blockDim.x / cq : 1;   // CTAs of up to 256 threads: one group
    const int t = MAXT > 256 ? tid % cq : tid, rg = MAXT > 256 ? tid / cq : 0;
    const int ch = 4 * t;
    extern __shared__ float4 xb[];             // [2][blockDim.x] when R > 1 (dynamic, compress_smem)
    const int nt = (int)blockDim.x;

    // pass 1: per-channel max of the logits
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 8
    for (int j = rg; j < m; j += R) {
        float4 z = load4<T>(cur_z + (int64_t)j * c + ch);
        float4 b = load4_bias(ba, (int64_t)j * c + ch);
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], f4get(z, k) + f4get(b, k));
    }
    if (hz) {
#pragma unroll 8
        for (int j = rg; j < m; j += R) {
            float4 z = load4<T>(hz + (int64_t)j * c + ch);
            float4 b = load4_bias(bb, (int64_t)j * c + ch);
#pragma unroll
            for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], f4get(z, k) + f4get(b, k));
        }
    }
    if (R > 1) {
        xb[tid] = make_float4(mx[0], mx[1], mx[2], mx[3]);
        __syncthreads();
        for (int g = 0; g < R; ++g) {
            const float4 o = xb[g * cq + t];
            mx[0] = fmaxf(mx[0], o.x);
            mx[1] = fmaxf(mx[1], o.y);
            mx[2] = fmaxf(mx[2], o.z);
            mx[3] = fmaxf(mx[3], o.w);
        }
    }
    // pass 2: softmax-weighted sum
    float num[4] = {0.f, 0.f, 0.f, 0.f}, den[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = rg; j < m; j += R) {
        float4 z = load4<T>(cur_z + (int64_t)j * c + ch);
        float4 b = load4_bias(ba, (int64_t)j * c + ch);
        float4 v = load4<T>(cur_c + (int64_t)j * c + ch);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float e = expf(f4get(z, k) + f4get(b, k) - mx[k]);
            den[k] += e;
            num[k] = fmaf(e, f4get(v, k), num[k]);
        }
    }
    if (hz) {
#pragma unroll 8
        for (int j = rg; j < m; j += R) {
            float4 z = load4<T>(hz + (int64_t)j * c + ch);
            float4 b = load4_bias(bb, (int64_t)j * c + ch);
            float4 v = load4<T>(hc + (int64_t)j * c + ch);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float e = expf(f4get(z, k) + f4get(b, k) - mx[k]);
                den[k] += e;
                num[k] = fmaf(e, f4get(v, k), num[k]);
            }
        }
    }
    if (R > 1) {
        // group partials in group order (xb's first half is free: every thread has
        // read the maxima before it passed this barrier)
        __syncthreads();
        xb[tid] = make_float4(num[0], num[1], num[2], num[3]);
        xb[nt + tid] = make_float4(den[0], den[1], den[2], den[3]);
        __syncthreads();
        float4 n4 = xb[t], d4 = xb[nt + t];
        for (int g = 1; g < R; ++g) {
            const float4 o = xb[g * cq + t], e = xb[nt + g * cq + t];
            n4.x += o.x; n4.y += o.y; n4.z += o.z; n4.w += o.w;
            d4.x += e.x; d4.y += e.y; d4.z += e.z; d4.w += e.w;
        }
        num[0] = n4.x; num[1] = n4.y; num[2] = n4.z; num[3] = n4.w;
        den[0] = d4.x; den[1] = d4.y; den[2] = d4.z; den[3] = d4.w;
    }
    float y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = num[k] / den[k];

    // RMSNorm over the c channels of the entry (row group 0 holds the entry; the other
    // groups only take part in the barriers)
    if (flags & CSA2_W_NORM) {
        __shared__ float red[32];
        float ss = rg == 0 ? y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3] : 0.0f;
        ss = warp_sum(ss);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        if (tid < 32) {
            float v = (tid < (int)(blockDim.x >> 5)) ? red[tid] : 0.f;
            v = warp_sum(v);
            if (tid == 0) red[0] = v;
        }
        __syncthreads();
        float r = 1.0f / sqrtf(red[0] / (float)c + 1e-6f);
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] *= r;
    }
    if (rg != 0) return;
    // RoPE on the last 64 channels (interleaved pairs) at the entry's position
    if ((flags & CSA2_W_ROPE) && ch >= c - 64) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            int j = (ch + 2 * p - (c - 64)) >> 1;
            float cs, sn;
            rope_cos_sin(rope, pos, j, cs, sn);
            float x0 = y[2 * p], x1 = y[2 * p + 1];
            y[2 * p] = x0 * cs - x1 * sn;
            y[2 * p + 1] = x0 * sn + x1 * cs;
        }
    }
    // store
    if (OUT == OUT_F32) {
        float* o = reinterpret_cast<float*>(out) + orow * (int64_t)c + ch;
        *reinterpret_cast<float4*>(o) = make_float4(y[0], y[1], y[2], y[3]);
    } else if (OUT == OUT_BF16) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + orow * (int64_t)c + ch;
        uint2 u;
        u.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y[0])) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y[1])) << 16);
        u.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y[2])) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y[3])) << 16);
        *reinterpret_cast<uint2*>(o) = u;
    } else if (OUT == OUT_FP4) {
        // FP4: the 16-channel group is lanes 4g..4g+3 of this warp
        float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        uint32_t sb = e4m3_byte(__fdiv_rn(amax, 6.0f));
        float s = e4m3_to_f32(sb);
        uint32_t codes = 0;
        if (s != 0.0f)
            codes = e2m1x2(__fdiv_rn(y[0], s), __fdiv_rn(y[1], s)) |
                    (e2m1x2(__fdiv_rn(y[2], s), __fdiv_rn(y[3], s)) << 8);
        uint8_t* row = reinterpret_cast<uint8_t*>(out) + orow * fp4_row_bytes(c);
        *reinterpret_cast<uint16_t*>(row + ch / 2) = (uint16_t)codes;
        if ((t & 3) == 0) row[c / 2 + ch / 16] = (uint8_t)sb;
    } else {
        // MXFP4: the 32-channel group is lanes 8g..8g+7 of this warp
        float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const uint32_t code = mx_scale_code(amax);
        uint32_t codes = 0;
        if (amax > 0.0f) {
            const float X = e8m0_to_f32(code);
            codes = e2m1x2(__fdiv_rn(y[0], X), __fdiv_rn(y[1], X)) | (e2m1x2(__fdiv_rn(y[2], X), __fdiv_rn(y[3], X)) << 8);
        }
        uint8_t* row = reinterpret_cast<uint8_t*>(out) + orow * mxfp4_row_bytes(c);
        *reinterpret_cast<uint16_t*>(row + ch / 2) = (uint16_t)codes;
        if ((t & 7) == 0) row[c / 2 + ch / 32] = (uint8_t)code;
    }
}

template <typename T, int OUT, int MAXT>
__global__ void __launch_bounds__(MAXT) compress_kernel(
    const T* __restrict__ ca, const T* __restrict__ za, const T* __restrict__ cb,
    const T* __restrict__ zb, const float* __restrict__ ba, const float* __restrict__ bb,
    const T* __restrict__ prev_cb, const T* __restrict__ prev_zb, int64_t n_tokens, int c, int m,
    const int64_t* __restrict__ pos0_arr, const RopeTable rope, unsigned flags, void* __restrict__ out,
    int64_t out_seq_stride) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = blockIdx.x;            // entry within the stream
    const int64_t bseq = blockIdx.y;         // stream (sequence)
    const bool overlap = cb != nullptr;
    const int64_t in_off = bseq * n_tokens * (int64_t)c;
    ca += in_off;
    za += in_off;
    if (overlap) {
        cb += in_off;
        zb += in_off;
    }
    if (prev_cb) {
        prev_cb += bseq * (int64_t)m * c;
        prev_zb += bseq * (int64_t)m * c;
    }
    // history rows: block i-1 of (cb, zb), or the carried state for block 0
    const T* hc = nullptr;
    const T* hz = nullptr;
    if (overlap) {
        if (i > 0) {
            hc = cb + (m * (i - 1)) * (int64_t)c;
            hz = zb + (m * (i - 1)) * (int64_t)c;
        } else if (prev_cb) {
            hc = prev_cb;
            hz = prev_zb;
        }
    }
    const int64_t pos = (pos0_arr ? pos0_arr[bseq] : 0) + (int64_t)m * i;
    compress_entry<T, OUT, MAXT>(ca + (m * i) * (int64_t)c, za + (m * i) * (int64_t)c, hc, hz, ba, bb, c, m, pos, rope,
                           flags, out, bseq * out_seq_stride + i);
}

// Packed samples (varlen): the tokens of S samples lie back to back in one stream,
// sample s at tokens cu_tokens[s] .. cu_tokens[s+1]-1.  Each sample is compressed on
// its own -- its blocks start at its first token, its first block has no history, and
// a tail shorter than m is left out rather than completed by the next sample's tokens
// (DSA-to-CSA/HCA page, the note under the compressor code and «算法语义») -- and
// entry i of sample s goes to row s*out_seq_stride + i at position pos0[s] + m*i.
// Grid: (max entries per sample, S); CTAs past their sample's entry count exit.
template <typename T, int OUT, int MAXT>
__global__ void __launch_bounds__(MAXT) compress_varlen_kernel(
    const T* __restrict__ ca, const T* __restrict__ za, const T* __restrict__ cb, const T* __restrict__ zb,
    const float* __restrict__ ba, const float* __restrict__ bb, const int64_t* __restrict__ cu_tokens, int c, int m,
    const int64_t* __restrict__ pos0_arr, const RopeTable rope, unsigned flags, void* __restrict__ out,
    int64_t out_seq_stride) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = blockIdx.x;
    const int64_t smp = blockIdx.y;
    const int64_t t0 = cu_tokens[smp], n = cu_tokens[smp + 1] - t0;
    if (i >= n / m) return;                  // the whole CTA: past this sample's complete blocks
    const bool overlap = cb != nullptr;
    const int64_t r0 = (t0 + m * i) * (int64_t)c;
    const T* hc = nullptr;
    const T* hz = nullptr;
    if (overlap && i > 0) {
        hc = cb + r0 - (int64_t)m * c;
        hz = zb + r0 - (int64_t)m * c;
    }
    const int64_t pos = (pos0_arr ? pos0_arr[smp] : 0) + (int64_t)m * i;
    compress_entry<T, OUT, MAXT>(ca + r0, za + r0, hc, hz, ba, bb, c, m, pos, rope, flags, out, smp * out_seq_stride + i);
}

// One decode step for B sequences (a CTA each): the token at position pos[b] (< 0: no
// token this step) is stored in slot pos % m of the state; when it completes block
// i = pos / m, entry i (position m*i) is written to row b*out_seq_stride + i of out
// and the block's overlap half becomes the history of block i+1.
// state per sequence: [ca, za (, cb, zb, prev cb, prev zb)] x [m, c] in T.
template <typename T, int OUT, int MAXT>
__global__ void __launch_bounds__(MAXT) compress_step_kernel(
    const T* __restrict__ ca, const T* __restrict__ za, const T* __restrict__ cb, const T* __restrict__ zb,
    const float* __restrict__ ba, const float* __restrict__ bb, const int64_t* __restrict__ pos_arr, T* state,
    int c, int m, const RopeTable rope, unsigned flags, void* __restrict__ out, int64_t out_seq_stride) {
    pdl_wait();
    pdl_trigger();
    const int64_t b = blockIdx.x;
    const int cq = c >> 2;
    const int R = MAXT > 256 ? (int)blockDim.x / cq : 1;
    const int rg = MAXT > 256 ? (int)threadIdx.x / cq : 0;
    const int ch = 4 * (MAXT > 256 ? (int)threadIdx.x % cq : (int)threadIdx.x);
    const bool overlap = cb != nullptr;
    const int64_t mc = (int64_t)m * c;
    T* st = state + b * (overlap ? 6 : 2) * mc;
    T* s_ca = st;
    T* s_za = st + mc;
    T* s_cb = st + 2 * mc;
    T* s_zb = st + 3 * mc;
    T* s_pcb = st + 4 * mc;
    T* s_pzb = st + 5 * mc;
    const int64_t p = pos_arr[b];
    if (p < 0) return;                       // the whole CTA: no token for this sequence
    const int j = (int)(p % m);
    const int64_t i = p / m;
    // row group 0 stores the token; each thread touches only its own 4 channels of a
    // row, and the rows of a group's turn below are read after the barrier
    if (rg == 0) {
        copy4<T>(s_ca + (int64_t)j * c + ch, ca + b * c + ch);
        copy4<T>(s_za + (int64_t)j * c + ch, za + b * c + ch);
        if (overlap) {
            copy4<T>(s_cb + (int64_t)j * c + ch, cb + b * c + ch);
            copy4<T>(s_zb + (int64_t)j * c + ch, zb + b * c + ch);
        }
    }
    if (j != m - 1) return;                  // the block is not complete yet
    if (R > 1) __syncthreads();
    const bool hist = overlap && i > 0;
    compress_entry<T, OUT, MAXT>(s_ca, s_za, hist ? s_pcb : nullptr, hist ? s_pzb : nullptr, ba, bb, c, m,
                           (int64_t)m * i, rope, flags, out, b * out_seq_stride + i);
    if (overlap) {
        // every group has passed compress_entry's last barrier, so the history rows
        // are read; the new block's rows were stored before the barrier above
        __syncthreads();
        for (int r = rg; r < m; r += R) {
            copy4<T>(s_pcb + (int64_t)r * c + ch, s_cb + (int64_t)r * c + ch);
            copy4<T>(s_pzb + (int64_t)r * c + ch, s_zb + (int64_t)r * c + ch);
        }
    }
}

template <typename T, int MAXT>
csa2_status launch_compress_t(const void* ca, const void* za, const void* cb, const void* zb,
                            const float* ba, const float* bb, const void* pcb, const void* pzb, int B,
                            int64_t n_tokens, int c, int m, const int64_t* pos0, float base, unsigned flags,
                            void* out, csa2_dtype out_dt, int64_t oss, cudaStream_t s) {
    dim3 grid((unsigned)(n_tokens / m), (unsigned)B), block((c / 4) * compress_row_groups(m, c));
    const RopeTable rope = make_rope_table(base);
    const T* a = (const T*)ca;
    const T* z = (const T*)za;
    const T* b = (const T*)cb;
    const T* zz = (const T*)zb;
    const T* p1 = (const T*)pcb;
    const T* p2 = (const T*)pzb;
    csa2_status r;
    if (out_dt == CSA2_F32)
        r = launch_pdl(compress_kernel<T, OUT_F32, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, p1, p2, n_tokens, c, m,
                       pos0, rope, flags, out, oss);
    else if (out_dt == CSA2_BF16)
        r = launch_pdl(compress_kernel<T, OUT_BF16, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, p1, p2, n_tokens, c, m,
                       pos0, rope, flags, out, oss);
    else if (out_dt == CSA2_FP4_E4M3x16)
        r = launch_pdl(compress_kernel<T, OUT_FP4, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, p1, p2, n_tokens, c, m,
                       pos0, rope, flags, out, oss);
    else
        r = launch_pdl(compress_kernel<T, OUT_MX, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, p1, p2, n_tokens, c, m,
                       pos0, rope, flags, out, oss);
    return r != CSA2_OK ? r : csa2_launch_status();
}

template <typename T, int MAXT>
csa2_status launch_varlen_t(const void* ca, const void* za, const void* cb, const void* zb, const float* ba,
                          const float* bb, const int64_t* cu_tokens, int S, int64_t max_entries, int c, int m,
                          const int64_t* pos0, float base, unsigned flags, void* out, csa2_dtype out_dt, int64_t oss,
                          cudaStream_t s) {
    const RopeTable rope = make_rope_table(base);
    const T* a = (const T*)ca;
    const T* z = (const T*)za;
    const T* b = (const T*)cb;
    const T* zz = (const T*)zb;
    const dim3 grid((unsigned)max_entries, (unsigned)S), block((c / 4) * compress_row_groups(m, c));
    csa2_status r;
    if (out_dt == CSA2_F32)
        r = launch_pdl(compress_varlen_kernel<T, OUT_F32, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, cu_tokens, c, m,
                       pos0, rope, flags, out, oss);
    else if (out_dt == CSA2_BF16)
        r = launch_pdl(compress_varlen_kernel<T, OUT_BF16, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, cu_tokens, c, m,
                       pos0, rope, flags, out, oss);
    else if (out_dt == CSA2_FP4_E4M3x16)
        r = launch_pdl(compress_varlen_kernel<T, OUT_FP4, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, cu_tokens, c, m,
                       pos0, rope, flags, out, oss);
    else
        r = launch_pdl(compress_varlen_kernel<T, OUT_MX, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, cu_tokens, c, m,
                       pos0, rope, flags, out, oss);
    return r != CSA2_OK ? r : csa2_launch_status();
}

template <typename T, int MAXT>
csa2_status launch_step_t(const void* ca, const void* za, const void* cb, const void* zb, const float* ba,
                        const float* bb, const int64_t* pos, void* state, int B, int c, int m, float base,
                        unsigned flags, void* out, csa2_dtype out_dt, int64_t oss, cudaStream_t s) {
    const RopeTable rope = make_rope_table(base);
    const T* a = (const T*)ca;
    const T* z = (const T*)za;
    const T* b = (const T*)cb;
    const T* zz = (const T*)zb;
    T* st = (T*)state;
    const dim3 grid((unsigned)B), block((c / 4) * compress_row_groups(m, c));
    csa2_status r;
    if (out_dt == CSA2_F32)
        r = launch_pdl(compress_step_kernel<T, OUT_F32, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, pos, st, c, m, rope,
                       flags, out, oss);
    else if (out_dt == CSA2_BF16)
        r = launch_pdl(compress_step_kernel<T, OUT_BF16, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, pos, st, c, m, rope,
                       flags, out, oss);
    else if (out_dt == CSA2_FP4_E4M3x16)
        r = launch_pdl(compress_step_kernel<T, OUT_FP4, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, pos, st, c, m, rope,
                       flags, out, oss);
    else
        r = launch_pdl(compress_step_kernel<T, OUT_MX, MAXT>, grid, block, compress_smem(m, c), s, a, z, b, zz, ba, bb, pos, st, c, m, rope,
                       flags, out, oss);
    return r != CSA2_OK ? r : csa2_launch_status();
}

template <typename T>
csa2_status launch_compress(const void* ca, const void* za, const void* cb, const void* zb,
                            const float* ba, const float* bb, const void* pcb, const void* pzb, int B,
                            int64_t n_tokens, int c, int m, const int64_t* pos0, float base, unsigned flags,
                            void* out, csa2_dtype out_dt, int64_t oss, cudaStream_t s) {
    // long blocks run their row groups in up to CMP_MAX_THREADS threads; one group keeps
    // the small CTA (and its register budget)
    return compress_row_groups(m, c) > 1 ? launch_compress_t<T, CMP_MAX_THREADS>(ca, za, cb, zb, ba, bb, pcb, pzb, B, n_tokens, c, m, pos0, base, flags, out, out_dt, oss, s) : launch_compress_t<T, 256>(ca, za, cb, zb, ba, bb, pcb, pzb, B, n_tokens, c, m, pos0, base, flags, out, out_dt, oss, s);
}

template <typename T>
csa2_status launch_varlen(const void* ca, const void* za, const void* cb, const void* zb, const float* ba,
                          const float* bb, const int64_t* cu_tokens, int S, int64_t max_entries, int c, int m,
                          const int64_t* pos0, float base, unsigned flags, void* out, csa2_dtype out_dt, int64_t oss,
                          cudaStream_t s) {
    // long blocks run their row groups in up to CMP_MAX_THREADS threads; one group keeps
    // the small CTA (and its register budget)
    return compress_row_groups(m, c) > 1 ? launch_varlen_t<T, CMP_MAX_THREADS>(ca, za, cb, zb, ba, bb, cu_tokens, S, max_entries, c, m, pos0, base, flags, out, out_dt, oss, s) : launch_varlen_t<T, 256>(ca, za, cb, zb, ba, bb, cu_tokens, S, max_entries, c, m, pos0, base, flags, out, out_dt, oss, s);
}

template <typename T>
csa2_status launch_step(const void* ca, const void* za, const void* cb, const void* zb, const float* ba,
                        const float* bb, const int64_t* pos, void* state, int B, int c, int m, float base,
                        unsigned flags, void* out, csa2_dtype out_dt, int64_t oss, cudaStream_t s) {
    // long blocks run their row groups in up to CMP_MAX_THREADS threads; one group keeps
    // the small CTA (and its register budget)
    return compress_row_groups(m, c) > 1 ? launch_step_t<T, CMP_MAX_THREADS>(ca, za, cb, zb, ba, bb, pos, state, B, c, m, base, flags, out, out_dt, oss, s) : launch_step_t<T, 256>(ca, za, cb, zb, ba, bb, pos, state, B, c, m, base, flags, out, out_dt, oss, s);
}

}  // namespace

extern "C" csa2_status csa2_compress(csa2_ctx* ctx, const void* ca, const void* za, const void* cb,
                                     const void* zb, csa2_dtype in_dt, const float* ba, const float* bb,
                                     const void* prev_cb, const void* prev_zb, int B, int64_t n_tokens, int c,
                                     int m, const int64_t* pos0, float rope_base, unsigned flags, void* out,
                                     csa2_dtype out_dt, int64_t out_seq_stride, void* stream) {
    if (!ctx || B < 0 || B > 65535 || n_tokens < 0 || m < 1 || c <= 0) return CSA2_ERR_INVALID_ARG;
    if (n_tokens % m) return CSA2_ERR_INVALID_ARG;
    if (c % 128 || c > 1024) return CSA2_ERR_INVALID_ARG;
    if ((cb == nullptr) != (zb == nullptr)) return CSA2_ERR_INVALID_ARG;
    if ((prev_cb == nullptr) != (prev_zb == nullptr)) return CSA2_ERR_INVALID_ARG;
    if (prev_cb && !cb) return CSA2_ERR_INVALID_ARG;
    if (flags & ~(CSA2_W_NORM | CSA2_W_ROPE)) return CSA2_ERR_INVALID_ARG;
    if (in_dt != CSA2_F32 && in_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (out_dt != CSA2_F32 && out_dt != CSA2_BF16 && out_dt != CSA2_FP4_E4M3x16 && out_dt != CSA2_MXFP4_E8M0x32)
        return CSA2_ERR_UNSUPPORTED;
    if (n_tokens == 0 || B == 0) return CSA2_OK;
    if (out_seq_stride < n_tokens / m && B > 1) return CSA2_ERR_INVALID_ARG;
    if (!ca || !za || !out) return CSA2_ERR_INVALID_ARG;
    const size_t va = in_dt == CSA2_F32 ? 16 : 8;
    if (!aligned(ca, va) || !aligned(za, va) || (cb && (!aligned(cb, va) || !aligned(zb, va))) ||
        (prev_cb && (!aligned(prev_cb, va) || !aligned(prev_zb, va))) || (ba && !aligned(ba, 16)) ||
        (bb && !aligned(bb, 16)) || !aligned(out, 16))
        return CSA2_ERR_INVALID_ARG;
    if (n_tokens / m > 0x7FFFFFFF) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (in_dt == CSA2_F32)
        return launch_compress<float>(ca, za, cb, zb, ba, bb, prev_cb, prev_zb, B, n_tokens, c, m, pos0, rope_base,
                                      flags, out, out_dt, out_seq_stride, s);
    return launch_compress<__nv_bfloat16>(ca, za, cb, zb, ba, bb, prev_cb, prev_zb, B, n_tokens, c, m, pos0,
                                          rope_base, flags, out, out_dt, out_seq_stride, s);
}

extern "C" size_t csa2_compress_state_bytes(int B, int c, int m, csa2_dtype in_dt, int overlap) {
    if (B <= 0 || c <= 0 || m < 1 || (in_dt != CSA2_F32 && in_dt != CSA2_BF16)) return 0;
    return (size_t)B * (overlap ? 6 : 2) * (size_t)m * c * (in_dt == CSA2_F32 ? 4 : 2);
}

extern "C" csa2_status csa2_compress_step(csa2_ctx* ctx, const void* ca, const void* za, const void* cb,
                                          const void* zb, csa2_dtype in_dt, const float* ba, const float* bb,
                                          int B, int c, int m, const int64_t* pos, void* state, float rope_base,
                                          unsigned flags, void* out, csa2_dtype out_dt, int64_t out_seq_stride,
                                          void* stream) {
    if (!ctx || B < 0 || B > 65535 || m < 1 || c <= 0) return CSA2_ERR_INVALID_ARG;
    if (c % 128 || c > 1024) return CSA2_ERR_INVALID_ARG;
    if ((cb == nullptr) != (zb == nullptr)) return CSA2_ERR_INVALID_ARG;
    if (flags & ~(CSA2_W_NORM | CSA2_W_ROPE)) return CSA2_ERR_INVALID_ARG;
    if (in_dt != CSA2_F32 && in_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (out_dt != CSA2_F32 && out_dt != CSA2_BF16 && out_dt != CSA2_FP4_E4M3x16 && out_dt != CSA2_MXFP4_E8M0x32)
        return CSA2_ERR_UNSUPPORTED;
    if (B == 0) return CSA2_OK;
    if (!ca || !za || !pos || !state || !out || out_seq_stride < 0) return CSA2_ERR_INVALID_ARG;
    const size_t va = in_dt == CSA2_F32 ? 16 : 8;
    if (!aligned(ca, va) || !aligned(za, va) || (cb && (!aligned(cb, va) || !aligned(zb, va))) ||
        !aligned(state, 16) || (ba && !aligned(ba, 16)) || (bb && !aligned(bb, 16)) || !aligned(out, 16))
        return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (in_dt == CSA2_F32)
        return launch_step<float>(ca, za, cb, zb, ba, bb, pos, state, B, c, m, rope_base, flags, out, out_dt,
                                  out_seq_stride, s);
    return launch_step<__nv_bfloat16>(ca, za, cb, zb, ba, bb, pos, state, B, c, m, rope_base, flags, out, out_dt,
                                      out_seq_stride, s);
}

extern "C" csa2_status csa2_compress_state_seed(csa2_ctx* ctx, const void* ca, const void* za, const void* cb,
                                                const void* zb, csa2_dtype in_dt, int B, int64_t n_tokens, int c,
                                                int m, void* state, void* stream) {
    if (!ctx || B < 0 || n_tokens < 0 || m < 1 || c <= 0) return CSA2_ERR_INVALID_ARG;
    if ((cb == nullptr) != (zb == nullptr)) return CSA2_ERR_INVALID_ARG;
    if (in_dt != CSA2_F32 && in_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (B == 0 || n_tokens == 0) return CSA2_OK;
    if (!ca || !za || !state) return CSA2_ERR_INVALID_ARG;
    const size_t es = in_dt == CSA2_F32 ? 4 : 2;
    const bool overlap = cb != nullptr;
    const size_t row = (size_t)c * es, mc = (size_t)m * row;
    const size_t spitch = (size_t)n_tokens * row, dpitch = (overlap ? 6 : 2) * mc;
    const int64_t full = n_tokens / m, tail = n_tokens % m;
    cudaStream_t s = as_stream(stream);
    uint8_t* st = reinterpret_cast<uint8_t*>(state);
    // the unfinished block's rows into slots 0 .. tail-1
    if (tail > 0) {
        const size_t off = (size_t)full * m * row, w = (size_t)tail * row;
        const void* src[4] = {ca, za, cb, zb};
        for (int k = 0; k < (overlap ? 4 : 2); ++k)
            CSA2_CHECK_CUDA(cudaMemcpy2DAsync(st + k * mc, dpitch, reinterpret_cast<const uint8_t*>(src[k]) + off,
                                              spitch, w, (size_t)B, cudaMemcpyDeviceToDevice, s));
    }
    // the last complete block's overlap half becomes the history
    if (overlap && full > 0) {
        const size_t off = (size_t)(full - 1) * m * row;
        CSA2_CHECK_CUDA(cudaMemcpy2DAsync(st + 4 * mc, dpitch, reinterpret_cast<const uint8_t*>(cb) + off, spitch, mc,
                                          (size_t)B, cudaMemcpyDeviceToDevice, s));
        CSA2_CHECK_CUDA(cudaMemcpy2DAsync(st + 5 * mc, dpitch, reinterpret_cast<const uint8_t*>(zb) + off, spitch, mc,
                                          (size_t)B, cudaMemcpyDeviceToDevice, s));
    }
    return CSA2_OK;
}

extern "C" csa2_status csa2_compress_varlen(csa2_ctx* ctx, const void* ca, const void* za, const void* cb,
                                            const void* zb, csa2_dtype in_dt, const float* ba, const float* bb,
                                            int S, const int64_t* cu_tokens, int64_t max_tokens, int c, int m,
                                            const int64_t* pos0, float rope_base, unsigned flags, void* out,
                                            csa2_dtype out_dt, int64_t out_seq_stride, void* stream) {
    if (!ctx || S < 0 || S > 65535 || max_tokens < 0 || m < 1 || c <= 0) return CSA2_ERR_INVALID_ARG;
    if (c % 128 || c > 1024) return CSA2_ERR_INVALID_ARG;
    if ((cb == nullptr) != (zb == nullptr)) return CSA2_ERR_INVALID_ARG;
    if (flags & ~(CSA2_W_NORM | CSA2_W_ROPE)) return CSA2_ERR_INVALID_ARG;
    if (in_dt != CSA2_F32 && in_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (out_dt != CSA2_F32 && out_dt != CSA2_BF16 && out_dt != CSA2_FP4_E4M3x16 && out_dt != CSA2_MXFP4_E8M0x32)
        return CSA2_ERR_UNSUPPORTED;
    const int64_t max_entries = max_tokens / m;
    if (S == 0 || max_entries == 0) return CSA2_OK;
    if (max_entries > 0x7FFFFFFF) return CSA2_ERR_INVALID_ARG;
    if (!ca || !za || !cu_tokens || !out || out_seq_stride < (S > 1 ? max_entries : 0)) return CSA2_ERR_INVALID_ARG;
    const size_t va = in_dt == CSA2_F32 ? 16 : 8;
    if (!aligned(ca, va) || !aligned(za, va) || (cb && (!aligned(cb, va) || !aligned(zb, va))) ||
        (ba && !aligned(ba, 16)) || (bb && !aligned(bb, 16)) || !aligned(out, 16))
        return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (in_dt == CSA2_F32)
        return launch_varlen<float>(ca, za, cb, zb, ba, bb, cu_tokens, S, max_entries, c, m, pos0, rope_base, flags,
                                    out, out_dt, out_seq_stride, s);
    return launch_varlen<__nv_bfloat16>(ca, za, cb, zb, ba, bb, cu_tokens, S, max_entries, c, m, pos0, rope_base,
                                        flags, out, out_dt, out_seq_stride, s);
}
