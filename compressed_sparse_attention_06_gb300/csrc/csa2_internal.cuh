// Internal helpers shared by the CSA2 kernel files (device and host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "csa2.h"

struct csa2_ctx {
    int device;
    int num_sms;
    unsigned int* status;   // device word: bit 0 = out-of-range index, bit 1 = timeout
    int stall_next;         // test hook: next tensor-core scan runs with a silent producer
    long long stall_budget; // wait budget (cycles) for that launch
    int cluster16;          // 16-CTA clusters of the selection kernel fit: -1 unknown, 0 no, 1 yes
    void* noalloc_scratch;  // device address of the allocation-free entry point's array (looked up
                            // on its first call with this context; NULL until then)
};

#define CSA2_DEVBIT_RANGE 1u
#define CSA2_DEVBIT_TIMEOUT 2u

#define CSA2_CHECK_CUDA(call)                                   \
    do {                                                        \
        cudaError_t e_ = (call);                                \
        if (e_ != cudaSuccess) return CSA2_ERR_CUDA;            \
    } while (0)

static inline csa2_status csa2_launch_status() {
    return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

static inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Programmatic dependent launch.  Kernels of the decode step are launched with
// launch_pdl so a kernel's CTAs can be scheduled while the previous kernel on the
// stream finishes; every such kernel calls pdl_wait() before its first global-memory
// access (read or write), which returns once the previous kernel has completed and its
// writes are visible, so stream order holds for every dependency.  pdl_trigger() lets
// the next kernel's CTAs be scheduled.  Both are no-ops for an ordinary launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static inline csa2_status launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

static inline bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void csa2_flag(unsigned int* st, unsigned bit) {
    if (st) atomicOr(st, bit);
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Order-preserving map of a float to uint32 (larger float -> larger key); -0.0 is
// folded onto +0.0 so the two compare equal.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

// RoPE angles.  theta_j = base^(-2j/64) for the 32 pairs of the last 64 dims; the
// table holds theta_j / (2 pi) in double, computed once on the host.  On the device
// the angle pos * theta_j is reduced exactly to a fractional turn in double (one
// multiply and a floor: (double)pos is exact and the subtraction is exact), and cos
// and sin of that turn are evaluated in float.  Double-precision transcendental
// calls are avoided: their throughput on this part is very low.
struct RopeTable {
    double turns[32];
};

static inline RopeTable make_rope_table(float base) {
    RopeTable t;
    for (int j = 0; j < 32; ++j) t.turns[j] = pow((double)base, -2.0 * (double)j / 64.0) / 6.283185307179586;
    return t;
}

__device__ __forceinline__ void rope_cos_sin(const RopeTable& rt, int64_t pos, int j, float& c, float& s) {
    double u = (double)pos * rt.turns[j];
    u -= floor(u);
    sincospif(2.0f * (float)u, &s, &c);
}

// E2M1 pair from two floats: RNE, saturating to +-6, sign kept; `lo` goes to the
// low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// E4M3 (satfinite, RNE) of one float, as a byte.
__device__ __forceinline__ uint32_t e4m3_byte(float x) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
    return (uint32_t)(r & 0xFF);
}

// E4M3 byte -> float (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t h2;
    unsigned short in = (unsigned short)(b & 0xFF);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// E8M0 byte -> float 2^(b-127) (exact, 2^-127 is a float subnormal).
// MXFP4 block scale (OCP MX): E8M0 code of 2^(floor(log2 amax) - 2), clamped to
// 0..254; amax == 0 (or not positive) gives code 0.
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
    if (!(amax > 0.0f)) return 0u;
    const uint32_t bits = __float_as_uint(amax);
    const int e = (int)((bits >> 23) & 0xFF);
    const int fl = (e > 0) ? e - 127 : (31 - __clz((int)bits)) - 149;   // floor(log2 amax)
    const int cc = fl - 2 + 127;
    return (uint32_t)(cc < 0 ? 0 : (cc > 254 ? 254 : cc));
}

__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float((b & 0xFF) << 23);
}

// One MXFP4 block of 32 values (OCP MX): the E8M0 scale code (returned) and the 32
// E2M1 codes E2M1_RNE(x / X), X = 2^(code - 127), value 2i in the low nibble of byte i;
// all codes 0 when amax == 0.  X is a power of two, so x / X is taken as x * 2^(127 -
// code): that factor is exact in fp32 (2^-127 as a subnormal), and the product rounds
// exactly as the quotient would (the same real number, rounded once).
__device__ __forceinline__ uint32_t mxfp4_block32(const float (&v)[32], uint32_t (&w)[4]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t code = mx_scale_code(amax);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = 0u;
    if (amax > 0.0f) {
        const float rX = code == 254u ? __uint_as_float(0x00400000u) : __uint_as_float((254u - code) << 23);
#pragma unroll
        for (int i = 0; i < 32; i += 2) w[i / 8] |= e2m1x2(v[i] * rX, v[i + 1] * rX) << (4 * (i % 8));
    }
    return code;
}

// Magnitudes of the 8 E2M1 codes (format definition: 2 exponent bits with bias
// 1, one mantissa bit).
__device__ __forceinline__ float e2m1_to_f32(uint32_t nib) {
    uint32_t e = (nib >> 1) & 3u, mbit = nib & 1u;
    float mag = (e == 0) ? 0.5f * (float)mbit : ldexpf(1.0f + 0.5f * (float)mbit, (int)e - 1);
    return (nib & 8u) ? -mag : mag;
}

// Eight E2M1 codes (one 32-bit word, code 2i in the low nibble of byte i) -> f32,
// through the exact E2M1 -> f16 conversion.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float (&o)[8]) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(*reinterpret_cast<__half2*>(&h[i]));
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}

// Row bytes of the packed formats.
__host__ __device__ constexpr inline int64_t fp4_row_bytes(int c) { return c / 2 + c / 16; }
__host__ __device__ constexpr inline int64_t mxfp4_row_bytes(int d) { return d / 2 + d / 32; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
