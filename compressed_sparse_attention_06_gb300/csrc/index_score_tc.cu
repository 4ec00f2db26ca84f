// Tensor-core Lightning-indexer scan (tcgen05, sm_103a).
//
// Computes eq. (16) of the DSA-to-CSA/HCA page,
//     I[t, s] = sum_h w[t, h] * ReLU(q^I[t, h] . K^I[s]),
// for 64 indexer heads of 128 dims, over tiles of 128 entries, with the block max
// over 8 entries (CSA2 page, «解码器里的分层索引») fused into the epilogue, or over
// the pooled candidates of a Reindex layer.
//
// One MMA per 16-dim slice: D[128 entries x N] += A[128 entries x 16] * B[N x 16]^T
// with N = 64 heads x QT queries, D in tensor memory (fp32), kind::f16.
//
// Warp roles (320 threads):
//   warp 0     producer: bulk / TMA copies of key tiles into a shared-memory ring
//              (bf16 candidates: lanes 0-15 each copy one of the tile's 16 pooled
//              blocks, 2 KB, with a single 3-D tensor copy that lands both 64-dim
//              halves; one copy per half, 32 a tile, took 94 us for 64 x 16,384
//              candidates against 80 us, and one lane issuing them all 148 us)
//   warp 1     MMA issuer (one lane); owns the tensor-memory allocation
//   warps 2-5  converters (MXFP4 keys only): each thread takes one entry row of the
//              staged tile, turns its 128 E2M1 codes into f16 with the block scale
//              folded in, and writes the row into tensor memory (the MMA's A operand)
//   warps 6-9  epilogue: each thread reads its entry's N accumulators from tensor
//              memory, applies ReLU and the head weights, sums over heads, masks the
//              invisible entries, writes scores / the block max (8-lane shuffles).
//
// Exactness.  bf16 keys and queries go to the MMA unchanged (exact products, fp32
// accumulation).  MXFP4 keys are E2M1 x 2^k: the converter scales each row by
// 2^-rho (rho = largest block exponent - 13) so every value is an exact f16; the
// bf16 query of head h is scaled by 2^sigma_h (its largest element lands in
// [2^14, 2^15)) and converted to f16 -- exact for every element above 2^-31 of its
// head's maximum (below that, an error under 2^-40 of the maximum, far under the
// fp32 accumulation error).  The epilogue multiplies back by 2^(rho - sigma_h), an
// exact power-of-two rescale.  Blocks more than 2^36 below their row's largest
// block flush to zero, again far below the fp32 accumulation error.
//
// Every mbarrier wait is bounded; a wait that expires records CSA2_ERR_TIMEOUT and
// the CTA winds down (copies in flight are drained, tensor memory is freed).
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "index_score_tc.cuh"
#include "sm100_ptx.cuh"
#include "tma_host.cuh"

namespace {

using namespace sm100;

constexpr int TILE = 128;          // entries per tile (MMA M)
constexpr int DIM = 128;           // indexer head dim (MMA K in 8 steps of 16)
constexpr int HEADS = 64;          // indexer heads per query
constexpr int NTHREADS = 320;
constexpr int MX_ROW = 68;         // bytes of an MXFP4 row
constexpr int MX_STAGE = TILE * MX_ROW;     // 8704 B, a multiple of 16
constexpr int BF_STAGE = TILE * DIM * 2;    // 32 KB: two 16 KB K-chunks of 64 dims
constexpr long long WAIT_BUDGET = 1ll << 31;   // default wait limit, cycles (about a second)

enum KFmt { KF_MX = 0, KF_BF16 = 1 };

struct TcArgs {
    const __nv_bfloat16* q;       // [B, Q, 64, 128]
    const float* w;               // [B, Q, 64]
    const uint8_t* kmx;           // MXFP4 keys [B, N, 68]
    const int64_t* nv;            // [B, Q]
    const int32_t* pool;          // candidate mode: [B, Q, n_pool]
    float* scores;                // full: [B, Q, N]; candidate: [B, Q, n_pool*8]
    float* bmax;                  // full: [B, Q, ceil(N/8)]
    unsigned int* st;
    int B, Q, n_pool;
    int64_t N;
    int tiles;                    // tiles per query group
    int tiles_per_cta;
    long long budget;             // bounded-wait limit in cycles
    int stall;                    // test hook: the producer issues nothing
};

template <int KF, int QT>
struct Cfg {
    static constexpr int N = HEADS * QT;
    static constexpr int STAGES = KF == KF_MX ? 6 : 2;
    static constexpr int MIN_BLOCKS = QT == 1 ? 2 : 1;               // resident CTAs per SM we ask for
    static constexpr int STAGE_BYTES = KF == KF_MX ? MX_STAGE : BF_STAGE;
    static constexpr int B_BYTES = N * DIM * 2;                   // two K-chunks of N x 128 B
    static constexpr int A_COLS = KF == KF_MX ? 2 * 64 : 0;       // two f16 A buffers (64 cols each)
    static constexpr int D_COL0 = A_COLS;
    static constexpr int COLS_USED = A_COLS + 2 * N;
    static constexpr int TMEM_COLS = COLS_USED <= 32 ? 32 : COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128
                                   : COLS_USED <= 256 ? 256 : 512;
    // shared memory carve-up (offsets from a 1024-aligned base)
    static constexpr int OFF_B = 0;
    static constexpr int OFF_STAGE = B_BYTES;                        // multiple of 1024
    static constexpr int OFF_W = OFF_STAGE + STAGES * STAGE_BYTES;   // QT*64 floats
    static constexpr int OFF_RHO = OFF_W + QT * HEADS * 4;           // 4 x 128 ints
    static constexpr int OFF_BLK = OFF_RHO + 4 * TILE * 4;           // 2 x 16 candidate block ids (unused)
    static constexpr int OFF_BAR = ((OFF_BLK + 2 * 16 * 4) + 7) & ~7;
    static constexpr int N_BARS = 2 * STAGES + 8;
    static constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
    static constexpr int SMEM_NEED = OFF_TMEMPTR + 16 + 1024;        // + alignment slack
    // MXFP4: at least 80 KB so no more than two CTAs share an SM (2 x 256 TMEM columns)
    static constexpr int SMEM = (KF == KF_MX && SMEM_NEED < 80 * 1024) ? 80 * 1024 : SMEM_NEED;
    static_assert(COLS_USED <= 512, "tensor memory");
    static_assert(OFF_STAGE % 1024 == 0, "swizzle atoms need 1024-byte alignment");
    static_assert(KF == KF_MX || (BF_STAGE % 1024) == 0, "bf16 stages");
};

// f16 bits of 2^e for e <= 15 (subnormal below -14, zero below -24)
__device__ __forceinline__ uint32_t f16_pow2_bits(int e) {
    if (e >= -14) return (uint32_t)(e + 15) << 10;
    if (e >= -24) return 1u << (e + 24);
    return 0u;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Four E2M1 pairs (one 32-bit word of codes) -> four f16x2 words, exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t x, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(x));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int KF, int QT, bool CAND>
__global__ void __launch_bounds__(NTHREADS, Cfg<KF, QT>::MIN_BLOCKS) index_scan_tc_kernel(const TcArgs a,
                                                                  const __grid_constant__ CUtensorMap tmap_full,
                                                                  const __grid_constant__ CUtensorMap tmap_blk) {
    using C = Cfg<KF, QT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sB = smem + C::OFF_B;
    uint8_t* sStage = smem + C::OFF_STAGE;
    float* sW = reinterpret_cast<float*>(smem + C::OFF_W);
    int* sRho = reinterpret_cast<int*>(smem + C::OFF_RHO);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                          // [STAGES]
    uint64_t* empty = bars + C::STAGES;             // [STAGES]
    uint64_t* afull = bars + 2 * C::STAGES;         // [2]
    uint64_t* mdone = afull + 2;                    // [2]
    uint64_t* dempty = mdone + 2;                   // [2]
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMPTR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int groups_per_b = (a.Q + QT - 1) / QT;
    const int g = blockIdx.y;
    const int b = g / groups_per_b;
    const int q0 = (g % groups_per_b) * QT;
    int64_t V[QT];
    int64_t vmax = 0;
#pragma unroll
    for (int qi = 0; qi < QT; ++qi) {
        V[qi] = (q0 + qi < a.Q) ? a.nv[(int64_t)b * a.Q + q0 + qi] : 0;
        if (V[qi] > a.N && !CAND) V[qi] = a.N;
        vmax = V[qi] > vmax ? V[qi] : vmax;
    }
    // this CTA's tiles, and the active ones (some visible entry / candidate)
    const int t_begin = blockIdx.x * a.tiles_per_cta;
    const int t_end = min(a.tiles, t_begin + a.tiles_per_cta);
    int t_act_end = t_end;
    if (!CAND) t_act_end = min(t_end, (int)((vmax + TILE - 1) / TILE));
    const int n_act = max(0, t_act_end - t_begin);

    // ---- set-up: barriers, tensor memory, the B operand (queries) and head weights
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&full[i], (CAND && KF == KF_BF16) ? 32 : 1);
            mbar_init(&empty[i], KF == KF_MX ? 4 : 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&afull[j], 4);
            mbar_init(&mdone[j], 1);
            mbar_init(&dempty[j], 4);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sTmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    // queries: warp per (query, head) row; lane owns dims 4*lane .. 4*lane+3
    for (int r = warp; r < C::N; r += NTHREADS / 32) {
        const int qi = r / HEADS, h = r % HEADS;
        const bool qok = q0 + qi < a.Q;
        const int64_t qrow = ((int64_t)b * a.Q + q0 + qi) * HEADS + h;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (qok) {
            uint2 u = *reinterpret_cast<const uint2*>(a.q + qrow * DIM + 4 * lane);
            v[0] = __uint_as_float(u.x << 16);
            v[1] = __uint_as_float(u.x & 0xFFFF0000u);
            v[2] = __uint_as_float(u.y << 16);
            v[3] = __uint_as_float(u.y & 0xFFFF0000u);
        }
        uint32_t p0, p1;
        float wv = qok ? a.w[qrow] : 0.0f;
        if (KF == KF_MX) {
            float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
            m = warp_max(m);
            const int sigma = (m > 0.0f) ? 14 - ilogbf(m) : 0;
            p0 = pack_f16x2(ldexpf(v[0], sigma), ldexpf(v[1], sigma));
            p1 = pack_f16x2(ldexpf(v[2], sigma), ldexpf(v[3], sigma));
            wv = ldexpf(wv, -sigma);
        } else {
            uint2 u = make_uint2(0, 0);
            if (qok) u = *reinterpret_cast<const uint2*>(a.q + qrow * DIM + 4 * lane);
            p0 = u.x;
            p1 = u.y;
        }
        const int unit = lane >> 1;                  // 16-byte unit of 8 dims (0..15)
        const int kc = unit >> 3, uc = unit & 7;
        uint8_t* dst = sB + kc * (C::N * 128) + sw128_offset(r, uc) + (lane & 1) * 8;
        *reinterpret_cast<uint2*>(dst) = make_uint2(p0, p1);
        if (lane == 0) sW[r] = wv;
    }
    fence_proxy_async_smem();      // the MMA (async proxy) reads what the threads wrote
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    constexpr uint32_t IDESC = idesc_f16(TILE, C::N, KF == KF_BF16);
    bool ok = true;

    if (warp == 0) {
        // ============================ producer ============================
        if (CAND && KF == KF_BF16) {
            // 16 pooled blocks per tile: lane j < 16 copies block j whole (one 2 KB tensor
            // copy into [block j][half][8 rows x 128 B]), with its own arrival on the
            // stage barrier; lanes 16-31 and empty pool slots only arrive
            int issued = 0;
            const int j = lane & 15, hf = lane >> 4;
            const int64_t gq = (int64_t)b * a.Q + q0;
            for (int li = 0; li < (a.stall ? 0 : n_act); ++li) {
                const int s = li % C::STAGES, r = li / C::STAGES;
                const bool w = r == 0 || mbar_wait(&empty[s], (r - 1) & 1, a.budget, a.st);
                if (!__all_sync(0xffffffffu, w)) break;
                const int tile = t_begin + li;
                uint8_t* dst = sStage + s * C::STAGE_BYTES;
                const int64_t pi = (int64_t)tile * 16 + j;
                int32_t pb = pi < a.n_pool ? a.pool[gq * a.n_pool + pi] : -1;
                if (pb < 0 || (int64_t)pb * 8 + 8 > a.N) pb = -1;
                if (pb >= 0 && hf == 0) {
                    mbar_arrive_expect_tx(&full[s], 2048);
                    tma_load_3d(dst + j * 2048, &tmap_blk, 0, (int32_t)((int64_t)b * a.N + (int64_t)pb * 8), 0,
                                &full[s]);
                } else {
                    mbar_arrive(&full[s]);
                }
                ++issued;
            }
            if (lane == 0)
                for (int li = max(0, issued - C::STAGES); li < issued; ++li)
                    mbar_wait(&full[li % C::STAGES], (li / C::STAGES) & 1, a.budget, a.st);
        } else if (lane == 0) {
            int issued = 0;
            for (int li = 0; li < (a.stall ? 0 : n_act) && ok; ++li) {
                const int s = li % C::STAGES, r = li / C::STAGES;
                if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, a.budget, a.st)) { ok = false; break; }
                const int tile = t_begin + li;
                uint8_t* dst = sStage + s * C::STAGE_BYTES;
                const int64_t gq = (int64_t)b * a.Q + q0;      // first query row of the group
                if (!CAND) {
                    const int64_t row0 = (int64_t)tile * TILE;
                    if (KF == KF_MX) {
                        const int64_t rows = min((int64_t)TILE, a.N - row0);
                        const uint32_t bytes = (uint32_t)(rows * MX_ROW);
                        mbar_arrive_expect_tx(&full[s], bytes);
                        bulk_g2s(dst, a.kmx + ((int64_t)b * a.N + row0) * MX_ROW, bytes, &full[s]);
                    } else {
                        mbar_arrive_expect_tx(&full[s], BF_STAGE);
                        const int32_t y = (int32_t)((int64_t)b * a.N + row0);
                        tma_load_2d(dst, &tmap_full, 0, y, &full[s]);
                        tma_load_2d(dst + BF_STAGE / 2, &tmap_full, 64, y, &full[s]);
                    }
                } else if (KF == KF_MX) {
                    // 16 pooled blocks of 8 MXFP4 entries per tile (bf16 candidates take the
                    // 32-lane path above)
                    const int32_t* pl = a.pool + gq * a.n_pool + (int64_t)tile * 16;
                    int32_t blk[16];
                    uint32_t bytes = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        int32_t pb = ((int64_t)tile * 16 + j < a.n_pool) ? pl[j] : -1;
                        if (pb < 0 || (int64_t)pb * 8 + 8 > a.N) pb = -1;
                        blk[j] = pb;
                        if (pb >= 0) bytes += 8 * MX_ROW;
                    }
                    mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (blk[j] < 0) continue;
                        const int64_t row0 = (int64_t)b * a.N + (int64_t)blk[j] * 8;
                        bulk_g2s(dst + j * 8 * MX_ROW, a.kmx + row0 * MX_ROW, 8 * MX_ROW, &full[s]);
                    }
                }
                ++issued;
            }
            // drain: copies still in flight must land before the CTA can exit
            for (int li = max(0, issued - C::STAGES); li < issued; ++li)
                mbar_wait(&full[li % C::STAGES], (li / C::STAGES) & 1, a.budget, a.st);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            int done = 0;
            for (int li = 0; li < n_act && ok; ++li) {
                const int s = li % C::STAGES, r = li / C::STAGES;
                const int j = li & 1, u = li >> 1;
                if (KF == KF_MX) {
                    if (!mbar_wait(&afull[j], u & 1, a.budget, a.st)) { ok = false; break; }
                } else {
                    if (!mbar_wait(&full[s], r & 1, a.budget, a.st)) { ok = false; break; }
                }
                if (u > 0 && !mbar_wait(&dempty[j], (u - 1) & 1, a.budget, a.st)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem + C::D_COL0 + j * C::N;
                const uint32_t b_base = smem_u32(sB);
#pragma unroll
                for (int kk = 0; kk < DIM / 16; ++kk) {
                    const int kc = kk >> 2, ko = (kk & 3) * 32;
                    const uint64_t bdesc = sdesc_sw128(b_base + kc * (C::N * 128) + ko);
                    if (KF == KF_MX) {
                        mma_ts(d_tmem, tmem + j * 64 + kk * 8, bdesc, IDESC, kk > 0);
                    } else {
                        const uint32_t a_base = smem_u32(sStage + s * C::STAGE_BYTES);
                        // full tiles: K-chunk kc is 16 KB of 128 rows; pooled tiles: block j's
                        // chunk kc is the 1 KB atom at 2 KB j + 1 KB kc
                        const uint64_t adesc = CAND ? sdesc_sw128_sbo(a_base + kc * 1024 + ko, 2048)
                                                    : sdesc_sw128(a_base + kc * (BF_STAGE / 2) + ko);
                        mma_ss(d_tmem, adesc, bdesc, IDESC, kk > 0);
                    }
                }
                if (KF == KF_BF16) mma_commit(&empty[s]);
                mma_commit(&mdone[j]);
                ++done;
            }
            // the last MMAs must finish before tensor memory is released
            if (done > 0) mbar_wait(&mdone[(done - 1) & 1], ((done - 1) >> 1) & 1, a.budget, a.st);
        }
    } else if (warp < 6) {
        // ============================ converters (MXFP4) ============================
        if (KF == KF_MX) {
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;
            for (int li = 0; li < n_act; ++li) {
                const int s = li % C::STAGES, r = li / C::STAGES;
                const int j = li & 1, u = li >> 1;
                if (!mbar_wait(&full[s], r & 1, a.budget, a.st)) break;
                if (u > 0 && !mbar_wait(&mdone[j], (u - 1) & 1, a.budget, a.st)) break;
                tc_fence_after();     // the MMA that last read A[j] has completed
                const uint32_t* src = reinterpret_cast<const uint32_t*>(sStage + s * C::STAGE_BYTES + row * MX_ROW);
                uint32_t cw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) cw[i] = src[i];
                const uint32_t sw = src[16];
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                const int e0 = (int)(sw & 0xFF), e1 = (int)((sw >> 8) & 0xFF), e2 = (int)((sw >> 16) & 0xFF),
                          e3 = (int)(sw >> 24);
                const int emax = max(max(e0, e1), max(e2, e3));
                // block exponent relative to the row's largest block, which lands at 2^13
                // the four block multipliers, each as a pair of f16 lanes
                uint32_t m2[4];
                {
                    const uint32_t b0 = f16_pow2_bits(e0 - emax + 13), b1 = f16_pow2_bits(e1 - emax + 13),
                                   b2 = f16_pow2_bits(e2 - emax + 13), b3 = f16_pow2_bits(e3 - emax + 13);
                    m2[0] = b0 | (b0 << 16);
                    m2[1] = b1 | (b1 << 16);
                    m2[2] = b2 | (b2 << 16);
                    m2[3] = b3 | (b3 << 16);
                }
                sRho[(li & 3) * TILE + row] = emax - 127 - 13;
                uint32_t out[32];
                const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + j * 64;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {
                        const int wd = half * 8 + wi;
                        const uint32_t m2x = m2[wd >> 2];
                        uint32_t o0, o1, o2, o3;
                        e2m1x8_to_f16x2(cw[wd], o0, o1, o2, o3);
                        out[4 * wi + 0] = hmul2(o0, m2x);
                        out[4 * wi + 1] = hmul2(o1, m2x);
                        out[4 * wi + 2] = hmul2(o2, m2x);
                        out[4 * wi + 3] = hmul2(o3, m2x);
                    }
                    tmem_st32(tbase + half * 32, out);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[j]);
            }
        }
    } else {
        // ============================ epilogue ============================
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int64_t n_elems = CAND ? (int64_t)a.n_pool * 8 : a.N;
        const int64_t nb = (a.N + 7) / 8;
        for (int li = 0; li < n_act; ++li) {
            const int j = li & 1, u = li >> 1;
            if (!mbar_wait(&mdone[j], u & 1, a.budget, a.st)) break;
            tc_fence_after();
            const int tile = t_begin + li;
            const int64_t e = (int64_t)tile * TILE + row;           // element (entry or candidate)
            int64_t sid = e;                                         // entry id
            if (CAND) {
                // same validity rule as the producer: a real block lying inside the cache
                const int64_t gq = (int64_t)b * a.Q + q0;
                const int64_t pi = e >> 3;
                const int32_t pb = pi < a.n_pool ? a.pool[gq * a.n_pool + pi] : -1;
                sid = (pb >= 0 && (int64_t)pb * 8 + 8 <= a.N) ? (int64_t)pb * 8 + (e & 7) : INT64_MAX;
            }
            const int rho = (KF == KF_MX) ? sRho[(li & 3) * TILE + row] : 0;
            float sc[QT];
#pragma unroll
            for (int qi = 0; qi < QT; ++qi) {
                uint32_t d0[32], d1[32];
                const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + C::D_COL0 + j * C::N + qi * HEADS;
                tmem_ld32(tb, d0);
                tmem_ld32(tb + 32, d1);
                tmem_wait_ld();
                // four independent chains (head h feeds chain h mod 4) of w_h * 2 ReLU(d_h):
                // d + |d| is exactly 2 ReLU(d) (one add on the FMA pipe), and the final
                // halving is exact, so the sum equals the one of w_h * ReLU(d_h)
                float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                const float4* w4 = reinterpret_cast<const float4*>(sW + qi * HEADS);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 wv = w4[i];
                    const uint32_t* dd = i < 8 ? d0 : d1;
                    const int o = (i & 7) * 4;
                    const float x0 = __uint_as_float(dd[o]), x1 = __uint_as_float(dd[o + 1]);
                    const float x2 = __uint_as_float(dd[o + 2]), x3 = __uint_as_float(dd[o + 3]);
                    a4[0] = fmaf(wv.x, x0 + fabsf(x0), a4[0]);
                    a4[1] = fmaf(wv.y, x1 + fabsf(x1), a4[1]);
                    a4[2] = fmaf(wv.z, x2 + fabsf(x2), a4[2]);
                    a4[3] = fmaf(wv.w, x3 + fabsf(x3), a4[3]);
                }
                float acc = ((a4[0] + a4[1]) + (a4[2] + a4[3])) * 0.5f;
                if (KF == KF_MX)      // exact power-of-two rescale (2^rho built from its bits when normal)
                    acc = (rho >= -126 && rho <= 127) ? acc * __int_as_float((rho + 127) << 23) : ldexpf(acc, rho);
                const bool vis = sid < V[qi] && e < n_elems;
                sc[qi] = vis ? acc : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[j]);
#pragma unroll
            for (int qi = 0; qi < QT; ++qi) {
                if (q0 + qi >= a.Q) continue;
                const int64_t bq = (int64_t)b * a.Q + q0 + qi;
                if (a.scores && e < n_elems) a.scores[bq * n_elems + e] = sc[qi];
                if (!CAND && a.bmax) {
                    float m = sc[qi];
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    if ((lane & 7) == 0 && (e >> 3) < nb) a.bmax[bq * nb + (e >> 3)] = m;
                }
            }
        }
        // tiles of this CTA beyond every visible entry: -inf outputs
        for (int tile = t_begin + n_act; tile < t_end; ++tile) {
            const int64_t e = (int64_t)tile * TILE + row;
#pragma unroll
            for (int qi = 0; qi < QT; ++qi) {
                if (q0 + qi >= a.Q) continue;
                const int64_t bq = (int64_t)b * a.Q + q0 + qi;
                if (a.scores && e < n_elems) a.scores[bq * n_elems + e] = -INFINITY;
                if (!CAND && a.bmax && (lane & 7) == 0 && (e >> 3) < nb) a.bmax[bq * nb + (e >> 3)] = -INFINITY;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- host side
// 2-D map over bf16 rows of 128 values: box of 64 values x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
    return csa2_make_bf16_map(m, base, rows, DIM, 64, box_rows);
}

template <int KF, int QT, bool CAND>
csa2_status launch_tc(csa2_ctx* ctx, TcArgs& a, const void* kbf, cudaStream_t s) {
    using C = Cfg<KF, QT>;
    auto kern = index_scan_tc_kernel<KF, QT, CAND>;
    static int occ = 0;     // resident CTAs per SM for this variant
    if (occ == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
            return CSA2_ERR_CUDA;
        // residency from registers, shared memory and the 512 tensor-memory columns
        cudaFuncAttributes fa;
        int smem_sm = 0, regs_sm = 0, dev = 0;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess)
            return CSA2_ERR_CUDA;
        const int warp_regs = ((fa.numRegs * 32 + 255) / 256) * 256;      // allocation unit of 256 per warp
        const int by_regs = regs_sm / (warp_regs * (NTHREADS / 32));
        const int by_smem = smem_sm / (C::SMEM + 1024);                     // + per-CTA reserved shared memory
        occ = std::max(1, std::min(std::min(by_regs, by_smem), 512 / C::TMEM_COLS));
    }
    CUtensorMap mfull, mblk;
    memset(&mfull, 0, sizeof(mfull));
    memset(&mblk, 0, sizeof(mblk));
    // full scans read 128-row tiles, pooled candidates 8-row blocks whole (a 3-D map
    // whose halves' stride, 128 B, is below the rows' 256 B: the two dimensions never
    // address the same element, and the encoder takes it; were it refused, the call
    // would report CSA2_ERR_CUDA)
    if (KF == KF_BF16) {
        if (CAND ? !csa2_make_bf16_block_map(&mblk, kbf, (int64_t)a.B * a.N, 8)
                 : !make_map(&mfull, kbf, (int64_t)a.B * a.N, TILE))
            return CSA2_ERR_CUDA;
    }
    const int groups = a.B * ((a.Q + QT - 1) / QT);
    int64_t target = (int64_t)ctx->num_sms * occ;
    int splits = (int)std::min<int64_t>(a.tiles, std::max<int64_t>(1, (target + groups - 1) / groups));
    a.tiles_per_cta = (a.tiles + splits - 1) / splits;
    splits = (a.tiles + a.tiles_per_cta - 1) / a.tiles_per_cta;
    dim3 grid((unsigned)splits, (unsigned)groups);
    kern<<<grid, NTHREADS, C::SMEM, s>>>(a, mfull, mblk);
    return csa2_launch_status();
}

}  // namespace

csa2_status index_score_tc_dispatch(csa2_ctx* ctx, const void* q_idx, const float* w, const void* k_idx,
                                    csa2_dtype k_dt, int B, int Q, int64_t N, int H_I, const int64_t* n_visible,
                                    const int32_t* pool, int n_pool, int block, float* scores, float* block_max,
                                    cudaStream_t s) {
    if (H_I != HEADS || block != 8 || (N % 8) != 0 || N == 0) return CSA2_ERR_UNSUPPORTED;
    if (k_dt != CSA2_MXFP4_E8M0x32 && k_dt != CSA2_BF16) return CSA2_ERR_UNSUPPORTED;
    if ((int64_t)B * N > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED;      // tensor-map row coordinate
    if (pool && (n_pool % 16) != 0) return CSA2_ERR_UNSUPPORTED;
    TcArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16*>(q_idx);
    a.w = w;
    a.kmx = reinterpret_cast<const uint8_t*>(k_idx);
    a.nv = n_visible;
    a.pool = pool;
    a.scores = scores;
    a.bmax = block_max;
    a.st = ctx->status;
    a.B = B;
    a.Q = Q;
    a.N = N;
    a.n_pool = n_pool;
    a.tiles_per_cta = 0;
    a.budget = WAIT_BUDGET;
    a.stall = 0;
    if (ctx->stall_next) {
        a.stall = 1;
        if (ctx->stall_budget > 0) a.budget = ctx->stall_budget;
        ctx->stall_next = 0;
    }
    if (pool) {
        a.tiles = n_pool / 16;
    } else {
        a.tiles = (int)((N + TILE - 1) / TILE);
    }
    if (a.tiles == 0) return CSA2_OK;
    const bool mx = k_dt == CSA2_MXFP4_E8M0x32;
    // several queries of a sequence share one key tile (N = 256) for bf16 full scans;
    // candidate mode has one pool per query
    const int QT = (Q >= 4 && !mx && !pool) ? 4 : 1;
    if (mx) {
        return pool ? launch_tc<KF_MX, 1, true>(ctx, a, nullptr, s) : launch_tc<KF_MX, 1, false>(ctx, a, nullptr, s);
    }
    if (QT == 4)
        return pool ? launch_tc<KF_BF16, 4, true>(ctx, a, k_idx, s) : launch_tc<KF_BF16, 4, false>(ctx, a, k_idx, s);
    return pool ? launch_tc<KF_BF16, 1, true>(ctx, a, k_idx, s) : launch_tc<KF_BF16, 1, false>(ctx, a, k_idx, s);
}
