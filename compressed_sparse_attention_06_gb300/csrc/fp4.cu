// FP4 cache formats: pack / unpack kernels and their C-ABI entry points.
//
// FP4 main KV (CSA2 page, «890 字节是怎么来的»): one E4M3 scale per 16 channels,
// s = E4M3_RNE(amax / 6) (IEEE f32 division, satfinite); s == 0 -> codes 0; each
// code = E2M1_RNE(x / s) saturating at +-6.  Row = c/2 code bytes (channel 2i in
// the low nibble of byte i) then c/16 scale bytes.
// MXFP4 indexer K (same section; OCP MX rule): one E8M0 scale per 32 values,
// X = 2^(floor(log2 amax) - 2); amax == 0 -> scale byte 0 and codes 0; code =
// E2M1_RNE(x / X).  Row = d/2 code bytes then d/32 scale bytes.
#include "csa2_internal.cuh"

namespace {

// One thread per 16-channel group.
template <typename T>
__global__ void fp4_pack_kernel(const T* __restrict__ x, int64_t rows, int c, uint8_t* __restrict__ out,
                                int64_t out_ld) {
    pdl_wait();
    pdl_trigger();
    const int gpr = c / 16;
    int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= rows * gpr) return;
    int64_t r = g / gpr;
    int gi = (int)(g % gpr);
    const T* src = x + r * c + gi * 16;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = to_f32<T>(src[i]);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    uint32_t sb = e4m3_byte(__fdiv_rn(amax, 6.0f));
    float s = e4m3_to_f32(sb);
    uint32_t w0 = 0, w1 = 0;
    if (s != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            w0 |= e2m1x2(__fdiv_rn(v[i], s), __fdiv_rn(v[i + 1], s)) << (4 * i);
            w1 |= e2m1x2(__fdiv_rn(v[8 + i], s), __fdiv_rn(v[8 + i + 1], s)) << (4 * i);
        }
    }
    uint8_t* row = out + r * out_ld;
    uint32_t* codes = reinterpret_cast<uint32_t*>(row + gi * 8);   // rows are 4-byte aligned
    codes[0] = w0;
    codes[1] = w1;
    row[c / 2 + gi] = (uint8_t)sb;
}

// One thread per 32-value group.
template <typename T>
__global__ void mxfp4_pack_kernel(const T* __restrict__ x, int64_t rows, int d, uint8_t* __restrict__ out,
                                  int64_t out_ld) {
    pdl_wait();
    pdl_trigger();
    const int gpr = d / 32;
    int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= rows * gpr) return;
    int64_t r = g / gpr;
    int gi = (int)(g % gpr);
    const T* src = x + r * d + gi * 32;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = to_f32<T>(src[i]);
    uint32_t w[4];
    const uint32_t code = mxfp4_block32(v, w);
    uint8_t* row = out + r * out_ld;
    uint32_t* codes = reinterpret_cast<uint32_t*>(row + gi * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) codes[i] = w[i];
    row[d / 2 + gi] = (uint8_t)code;
}

template <typename T>
__global__ void fp4_unpack_kernel(const uint8_t* __restrict__ in, int64_t rows, int c, int group,
                                  bool mx, T* __restrict__ out) {
    const int gpr = c / group;
    int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= rows * gpr) return;
    int64_t r = g / gpr;
    int gi = (int)(g % gpr);
    const int64_t rb = mx ? mxfp4_row_bytes(c) : fp4_row_bytes(c);
    const uint8_t* row = in + r * rb;
    uint32_t sb = row[c / 2 + gi];
    float s = mx ? e8m0_to_f32(sb) : e4m3_to_f32(sb);
    const uint8_t* codes = row + gi * (group / 2);
    T* dst = out + r * c + gi * group;
    for (int i = 0; i < group / 2; ++i) {
        uint32_t b = codes[i];
        dst[2 * i] = from_f32<T>(e2m1_to_f32(b & 0xF) * s);
        dst[2 * i + 1] = from_f32<T>(e2m1_to_f32(b >> 4) * s);
    }
}

}  // namespace

extern "C" csa2_status csa2_fp4_pack(csa2_ctx* ctx, const void* x, csa2_dtype x_dt, int64_t rows, int c,
                                     csa2_dtype fmt, uint8_t* out, int64_t out_ld, void* stream) {
    if (!ctx || rows < 0 || c <= 0 || out_ld < 0 || (out_ld % 4)) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (!x || !out) return CSA2_ERR_INVALID_ARG;
    if (x_dt != CSA2_F32 && x_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if (!aligned(out, 4)) return CSA2_ERR_INVALID_ARG;
    const int threads = 256;
    if (fmt == CSA2_FP4_E4M3x16) {
        if (c % 64) return CSA2_ERR_INVALID_ARG;   // keeps every row 4-byte aligned
        if (out_ld == 0) out_ld = fp4_row_bytes(c);
        if (out_ld < fp4_row_bytes(c)) return CSA2_ERR_INVALID_ARG;
        int64_t n = rows * (c / 16);
        dim3 grid((unsigned)((n + threads - 1) / threads));
        if (x_dt == CSA2_F32)
            return launch_pdl(fp4_pack_kernel<float>, dim3(grid), dim3(threads), 0, as_stream(stream), (const float*)x,
                              rows, c, out, out_ld);
        else
            return launch_pdl(fp4_pack_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0, as_stream(stream),
                              (const __nv_bfloat16*)x, rows, c, out, out_ld);
    } else if (fmt == CSA2_MXFP4_E8M0x32) {
        if (c % 128) return CSA2_ERR_INVALID_ARG;  // keeps every row 4-byte aligned
        if (out_ld == 0) out_ld = mxfp4_row_bytes(c);
        if (out_ld < mxfp4_row_bytes(c)) return CSA2_ERR_INVALID_ARG;
        int64_t n = rows * (c / 32);
        dim3 grid((unsigned)((n + threads - 1) / threads));
        if (x_dt == CSA2_F32)
            return launch_pdl(mxfp4_pack_kernel<float>, dim3(grid), dim3(threads), 0, as_stream(stream),
                              (const float*)x, rows, c, out, out_ld);
        else
            return launch_pdl(mxfp4_pack_kernel<__nv_bfloat16>, dim3(grid), dim3(threads), 0, as_stream(stream),
                              (const __nv_bfloat16*)x, rows, c, out, out_ld);
    } else {
        return CSA2_ERR_UNSUPPORTED;
    }
    return csa2_launch_status();
}

extern "C" csa2_status csa2_fp4_unpack(csa2_ctx* ctx, const uint8_t* in, csa2_dtype fmt, int64_t rows, int c,
                                       void* out, csa2_dtype out_dt, void* stream) {
    if (!ctx || rows < 0 || c <= 0) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (!in || !out) return CSA2_ERR_INVALID_ARG;
    int group;
    bool mx;
    if (fmt == CSA2_FP4_E4M3x16) { group = 16; mx = false; }
    else if (fmt == CSA2_MXFP4_E8M0x32) { group = 32; mx = true; }
    else return CSA2_ERR_UNSUPPORTED;
    if (c % group) return CSA2_ERR_INVALID_ARG;
    const int threads = 256;
    int64_t n = rows * (c / group);
    dim3 grid((unsigned)((n + threads - 1) / threads));
    if (out_dt == CSA2_F32)
        fp4_unpack_kernel<float><<<grid, threads, 0, as_stream(stream)>>>(in, rows, c, group, mx, (float*)out);
    else if (out_dt == CSA2_BF16)
        fp4_unpack_kernel<__nv_bfloat16><<<grid, threads, 0, as_stream(stream)>>>(in, rows, c, group, mx, (__nv_bfloat16*)out);
    else
        return CSA2_ERR_UNSUPPORTED;
    return csa2_launch_status();
}
