// Lightning-indexer scan with the QK product in FP4 (tcgen05 kind::mxf4, sm_103a).
//
// Computes eq. (16) of the DSA-to-CSA/HCA page,
//     I[t, s] = sum_h w[t, h] * ReLU(q^I[t, h] . K^I[s]),
// when both the indexer query and the indexer keys are MXFP4 (E2M1 codes, one E8M0
// scale per 32 dims): the page runs the indexer QK path in FP4 (section «Lightning
// Indexer：公式 (13)–(17)» and «系统收益从哪里来»), and the CSA2 page stores K^I as
// 64 code bytes + 4 scale bytes per entry.  The block-scaled MMA multiplies the FP4
// values with their scales applied, so no element is converted on the CUDA cores.
//
// The pipeline steps over tiles of 256 entries (two MMA sub-tiles of 128): every
// per-step synchronisation (waits, commits) is paid once per 256 entries.  Per
// sub-tile: D[128 entries x 64 heads] = sum over two K=64 steps of (A x SFA)(B x
// SFB)^T, A = the sub-tile's key codes (tensor memory, one entry per lane), B = the
// query's codes (shared memory), SFA / SFB their E8M0 scales in tensor memory, D in
// fp32 tensor memory.  The block max over 8 entries (CSA2 page, «解码器里的分层索引»)
// is fused into the epilogue, or the tile is a list of 32 pooled candidate blocks
// (Reindex).  On request each CTA ends by counting the leading 12 key bits of its
// visible block maxima into a per-row histogram, which the pool's selection starts
// from.
//
// One CTA per SM (the grid splits each query's tiles over the SMs), 22 warps:
//   warp 0       producer, into an 8-stage ring of tiles.  Full scan: a tile is
//                17408 contiguous bytes, one bulk copy with an evict-first L2 policy
//                (the keys are read once); four lanes issue them, lane p owning stages
//                p and p+4 (one issuing thread alone sustains well under the HBM read
//                rate).  Candidates: a tile is 32 blocks of 544 bytes;
//                each of the 32 lanes issues one 544-byte bulk copy with its own
//                expect-tx arrival on the stage barrier (an empty pool slot only
//                arrives).
//   warp 1       MMA issuer (one lane): 4 MMAs and one commit per tile; owns the
//                tensor-memory allocation
//   warps 2-9    two copy groups (alternate tiles): each thread stores the 16 code
//                words of its two entries (one per sub-tile) into tensor memory, and
//                the group stores the tile's scale bytes next to them
//   warps 10-21  three epilogue groups (tiles in turn): each thread reads its two
//                entries' 64 head dots, applies ReLU and the head weights (packed
//                f32x2 FMAs), sums, masks the invisible entries and writes the scores /
//                block max
// Tensor memory: 3 D tiles (128 columns), 3 A tiles (32), their scales (8), the
// query's scales (4) = 508 of 512 columns.
//
// Phase safety: every mbarrier is waited on in phase order by construction -- each
// ring stage belongs to one producer lane and one copy group (the stage count is a
// multiple of both), buffers >= groups, and the MMA lane waits in tile order -- so no
// waiter can ask for phase k+1 while phase k is still open (the parity test would
// pass early).
//
// Exactness: E2M1 x E2M1 products and their per-block sums are exact; each block sum
// is scaled by a power of two and accumulated in fp32.
//
// Every mbarrier wait is bounded; a wait that expires records CSA2_ERR_TIMEOUT and
// the CTA winds down (copies and MMAs in flight are drained, tensor memory is freed).
#include <algorithm>

#include "index_score_tc.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace sm100;

constexpr int SUB = 128;                     // entries per MMA (M)
constexpr int TILE = 2 * SUB;                // entries per pipeline step
constexpr int HEADS = 64;                    // indexer heads (MMA N)
constexpr int MX_ROW = 68;                   // bytes of an MXFP4 row of 128 dims
constexpr int CODE_BYTES = 64;
constexpr int MX_STAGE = TILE * MX_ROW;      // 17408 B, a multiple of 16
constexpr int BLOCKS_PER_TILE = TILE / 8;    // candidate blocks of 8 entries per tile
constexpr long long WAIT_BUDGET = 1ll << 31;

constexpr int CPY_GROUPS = 2, EPI_GROUPS = 3;
constexpr int NWARPS = 2 + 4 * CPY_GROUPS + 4 * EPI_GROUPS;
constexpr int THREADS = NWARPS * 32;
constexpr int STAGES = 8, BUFS = 3;          // ring stages; A / D buffers (same index)
constexpr int PROD_LANES = 4;                // bulk-copy issuers (full scan)
constexpr int B_BYTES = HEADS * CODE_BYTES;  // 4 KB
static_assert(STAGES % PROD_LANES == 0 && STAGES % CPY_GROUPS == 0, "stage ownership");
static_assert(BUFS >= CPY_GROUPS && BUFS >= EPI_GROUPS, "buffer phases");

// shared memory (offsets from a 128-byte aligned base)
constexpr int OFF_B = 0;
constexpr int OFF_STAGE = OFF_B + B_BYTES;
constexpr int OFF_W = OFF_STAGE + STAGES * MX_STAGE;
constexpr int OFF_QS = OFF_W + HEADS * 4;                // the query's scale bytes, packed here
constexpr int OFF_BAR = OFF_QS + HEADS * 4;
constexpr int N_BARS = 2 * STAGES + 3 * BUFS;
constexpr int OFF_TMEMPTR = OFF_BAR + N_BARS * 8;
constexpr int OFF_HIST = OFF_TMEMPTR + 16;               // [CSA2_BLOCK_HIST_BINS] block-max digit counts
constexpr int SMEM = OFF_HIST + CSA2_BLOCK_HIST_BINS * 4 + 128;
// tensor memory
constexpr uint32_t D_COL0 = 0;                          // D[j]: 2 sub-tiles x 64 columns
constexpr uint32_t A_COL0 = D_COL0 + BUFS * 128;        // A[j]: 2 x 16 columns (128 E2M1 per lane)
constexpr uint32_t SFA_COL0 = A_COL0 + BUFS * 32;       // SFA[j]: 2 x 4 columns
constexpr uint32_t SFB_COL = SFA_COL0 + BUFS * 8;
constexpr uint32_t TMEM_COLS = 512;
static_assert(SFB_COL + 4 <= TMEM_COLS, "tensor memory");
// more than half of the SM's shared memory: one CTA per SM, so the 512-column
// allocation never waits on another CTA
static_assert(SMEM > 114 * 1024 && SMEM <= 227 * 1024, "shared memory");
static_assert(OFF_STAGE % 16 == 0 && MX_STAGE % 16 == 0 && OFF_BAR % 8 == 0, "alignment");

struct FpArgs {
    const uint8_t* qmx;           // MXFP4 queries [B, Q, 64, 68], or NULL with qbf
    const __nv_bfloat16* qbf;     // bf16 queries [B, Q, 64, 128], packed to MXFP4 here (or NULL)
    uint8_t* qmx_out;             // with qbf: the packed queries [B, Q, 64, 68], or NULL
    const float* w;               // [B, Q, 64]
    const uint8_t* kmx;           // MXFP4 keys [B, N, 68]
    const int64_t* nv;            // [B, Q]
    const int32_t* pool;          // candidate mode: [B, Q, n_pool]
    float* scores;                // full: [B, Q, N]; candidate: [B, Q, n_pool*8]
    float* bmax;                  // full: [B, Q, ceil(N/8)]
    uint32_t* hist;               // full: [B, Q, CSA2_BLOCK_HIST_BINS] (zeroed before), or NULL
    unsigned int* st;
    int B, Q, n_pool;
    int64_t N;
    int tiles;                    // tiles per query
    int tiles_per_cta;
    long long budget;
    int stall;                    // test hook: the producer issues nothing
};

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// (a0, a1) = (w0 * x0 + a0, w1 * x1 + a1), one packed f32x2 FMA (each lane rounds
// like fmaf).
__device__ __forceinline__ void ffma2(float& a0, float& a1, float w0, float w1, float x0, float x1) {
    asm("{\n\t.reg .b64 acc, wv, xv;\n\t"
        "mov.b64 acc, {%0, %1};\n\t"
        "mov.b64 wv, {%2, %3};\n\t"
        "mov.b64 xv, {%4, %5};\n\t"
        "fma.rn.f32x2 acc, wv, xv, acc;\n\t"
        "mov.b64 {%0, %1}, acc;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

template <bool CAND>
__global__ void __launch_bounds__(THREADS, 1) index_scan_fp4_kernel(const FpArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
    uint8_t* sB = smem + OFF_B;
    uint8_t* sStage = smem + OFF_STAGE;
    float* sW = reinterpret_cast<float*>(smem + OFF_W);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;                   // [STAGES] rows landed
    uint64_t* empty = full + STAGES;         // [STAGES] rows read by a copy group
    uint64_t* afull = empty + STAGES;        // [BUFS] A tile + its scales stored
    uint64_t* done = afull + BUFS;           // [BUFS] the tile's MMAs completed: D ready, A free
    uint64_t* dempty = done + BUFS;          // [BUFS] D tile read by an epilogue group
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + OFF_TMEMPTR);
    uint32_t* sHist = reinterpret_cast<uint32_t*>(smem + OFF_HIST);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;                // b * Q + q
    const int b = g / a.Q;

    // setup that touches no global memory runs before the wait for the previous
    // kernel (which, like every kernel before it, has released its tensor memory by the
    // time these CTAs can start: a kernel lets its successor start only after its own
    // wait returned)
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], CAND ? 32 : 1);   // cp.async: one arrival per lane
            mbar_init(&empty[i], 4);
        }
        for (int j = 0; j < BUFS; ++j) {
            mbar_init(&afull[j], 4);
            mbar_init(&done[j], 1);
            mbar_init(&dempty[j], 4);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sTmem, TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();                              // inputs of the previous kernel are complete
    int64_t V = a.nv[g];
    if (!CAND && V > a.N) V = a.N;
    const int t_begin = blockIdx.x * a.tiles_per_cta;
    const int t_end = min(a.tiles, t_begin + a.tiles_per_cta);
    int t_act_end = t_end;
    if (!CAND) t_act_end = min(t_end, (int)((V + TILE - 1) / TILE));
    const int n_act = max(0, t_act_end - t_begin);
    __syncthreads();                         // the barrier initialisations are visible to every warp
    // the query is prepared by warps 1.. while the producer (warp 0) already streams
    // keys: the B tile (query codes, thread = (head h, 16-byte unit u = MX block u)), its
    // scale bytes (sQS, then tensor memory) and the head weights
    uint8_t* sQS = smem + OFF_QS;
    uint32_t tmem = 0u;
    if (warp != 0) {
        constexpr int NT = THREADS - 32;
        const int tq = threadIdx.x - 32;
        if (a.qbf) {
            // pack the bf16 query here, by the rule of csa2_fp4_pack (one MX block a thread)
            for (int t = tq; t < HEADS * 4; t += NT) {
                const int h = t >> 2, u = t & 3;
                const uint4* src = reinterpret_cast<const uint4*>(a.qbf + ((int64_t)g * HEADS + h) * 128 + u * 32);
                float v[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 p = src[i];
                    const uint32_t pw[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[8 * i + 2 * j] = __uint_as_float(pw[j] << 16);
                        v[8 * i + 2 * j + 1] = __uint_as_float(pw[j] & 0xFFFF0000u);
                    }
                }
                uint32_t w4[4];
                const uint32_t code = mxfp4_block32(v, w4);
                *reinterpret_cast<uint4*>(sB + kmajor64_offset(h, u)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                sQS[h * 4 + u] = (uint8_t)code;
                if (a.qmx_out && blockIdx.x == 0) {
                    uint8_t* dst = a.qmx_out + ((int64_t)g * HEADS + h) * MX_ROW;
#pragma unroll
                    for (int i = 0; i < 4; ++i) reinterpret_cast<uint32_t*>(dst + u * 16)[i] = w4[i];
                    dst[CODE_BYTES + u] = (uint8_t)code;
                }
            }
        } else {
            const uint8_t* qrow0 = a.qmx + (int64_t)g * HEADS * MX_ROW;
            for (int t = tq; t < HEADS * 4; t += NT) {
                const int h = t >> 2, u = t & 3;
                const uint8_t* src = qrow0 + h * MX_ROW + u * 16;
                *reinterpret_cast<uint4*>(sB + kmajor64_offset(h, u)) =
                    make_uint4(ld_u32(src), ld_u32(src + 4), ld_u32(src + 8), ld_u32(src + 12));
            }
            for (int h = tq; h < HEADS; h += NT) reinterpret_cast<uint32_t*>(sQS)[h] = ld_u32(qrow0 + h * MX_ROW + CODE_BYTES);
        }
        for (int h = tq; h < HEADS; h += NT) sW[h] = a.w[(int64_t)g * HEADS + h];
        fence_proxy_async_smem();
        tc_fence_before();
        bar_sync_named(1, NT);
        tc_fence_after();
        tmem = *sTmem;
        // query scales -> tensor memory (warps 4..7: warp w reaches lane quarter w % 4).
        // Scale-factor layout: the 32-bit cell at lane 32j' + l, column c + j holds the
        // four block scales of row 32j + l (the same in each lane quarter); the query has
        // 64 rows (heads), so columns c and c+1.
        if (warp >= 4 && warp < 8) {
            const uint32_t s0 = reinterpret_cast<const uint32_t*>(sQS)[lane];
            const uint32_t s1 = reinterpret_cast<const uint32_t*>(sQS)[lane + 32];
            tmem_st4(tmem + ((uint32_t)((warp & 3) * 32) << 16) + SFB_COL, s0, s1, 0u, 0u);
            tmem_wait_st();
        }
        tc_fence_before();
        bar_sync_named(1, NT);
        tc_fence_after();
    }

    if (warp == 0) {
        // ============================ producer ============================
        if (!CAND) {
            // lane p issues tiles p, p+PL, ... (so it alone uses stages p, p+PL, ...);
            // a bulk copy of rows*68 bytes (rows a multiple of 8: a multiple of 16 B)
            constexpr int PL = PROD_LANES;
            const uint64_t pol = policy_evict_first();
            if (lane < PL) {
                int last = -1;
                for (int li = lane; li < (a.stall ? 0 : n_act); li += PL) {
                    const int s = li % STAGES, r = li / STAGES;
                    if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, a.budget, a.st)) break;
                    const int64_t row0 = (int64_t)(t_begin + li) * TILE;
                    const uint32_t bytes = (uint32_t)(min((int64_t)TILE, a.N - row0) * MX_ROW);
                    mbar_arrive_expect_tx(&full[s], bytes);
                    bulk_g2s_hint(sStage + s * MX_STAGE, a.kmx + ((int64_t)b * a.N + row0) * MX_ROW, bytes, &full[s], pol);
                    last = li;
                }
                // no copy may still be writing shared memory when the CTA exits: wait
                // for this lane's tiles of the last STAGES (no later tile reuses their
                // stages, so their phases are unambiguous; earlier ones were consumed)
                for (int li = last; li >= 0 && li > n_act - 1 - STAGES; li -= PL)
                    mbar_wait(&full[li % STAGES], (li / STAGES) & 1, a.budget, a.st);
            }
        } else {
            // lane j copies candidate block j of each tile: its 8 rows are 544 contiguous
            // bytes (a multiple of 16, at a 16-byte aligned offset since N is a multiple
            // of 8) in one bulk copy; empty or out-of-range slots copy nothing (their
            // rows are masked in the epilogue) and only arrive
            int last = -1;
            for (int li = 0; li < (a.stall ? 0 : n_act); ++li) {
                const int s = li % STAGES, r = li / STAGES;
                const bool w = r == 0 || mbar_wait(&empty[s], (r - 1) & 1, a.budget, a.st);
                if (!__all_sync(0xffffffffu, w)) break;
                int32_t pb = a.pool[(int64_t)g * a.n_pool + (int64_t)(t_begin + li) * BLOCKS_PER_TILE + lane];
                if (pb < 0 || (int64_t)pb * 8 + 8 > a.N) pb = -1;
                if (pb >= 0) {
                    mbar_arrive_expect_tx(&full[s], 8 * MX_ROW);
                    bulk_g2s(sStage + s * MX_STAGE + lane * (8 * MX_ROW),
                             a.kmx + ((int64_t)b * a.N + (int64_t)pb * 8) * MX_ROW, 8 * MX_ROW, &full[s]);
                } else {
                    mbar_arrive(&full[s]);
                }
                last = li;
            }
            // no copy may still be writing shared memory when the CTA exits (the last
            // STAGES tiles hold distinct stages, so their phases are unambiguous)
            for (int li = last; li >= 0 && li > last - STAGES; --li)
                mbar_wait(&full[li % STAGES], (li / STAGES) & 1, a.budget, a.st);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            int issued = 0;
            const uint32_t b_base = smem_u32(sB);
            for (int li = 0; li < n_act; ++li) {
                const int j = li % BUFS, u = li / BUFS;
                if (!mbar_wait(&afull[j], u & 1, a.budget, a.st)) break;
                if (u > 0 && !mbar_wait(&dempty[j], (u - 1) & 1, a.budget, a.st)) break;
                tc_fence_after();
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        // K = 64 per step: A columns 8kk .. 8kk+7, B's 16-byte units 2kk,
                        // 2kk+1, scale bytes 2kk, 2kk+1
                        const uint64_t bd = sdesc_kmajor_none(b_base + kk * 256, 128, 512);
                        mma_mxf4_ts(tmem + D_COL0 + j * 128 + sub * 64, tmem + A_COL0 + j * 32 + sub * 16 + kk * 8, bd,
                                    idesc_mxf4(SUB, HEADS, 2 * kk, 2 * kk), tmem + SFA_COL0 + j * 8 + sub * 4,
                                    tmem + SFB_COL, kk);
                    }
                }
                mma_commit(&done[j]);
                ++issued;
            }
            // the last commit covers every MMA of this thread
            if (issued > 0) mbar_wait(&done[(issued - 1) % BUFS], ((issued - 1) / BUFS) & 1, a.budget, a.st);
        }
    } else if (warp < 2 + 4 * CPY_GROUPS) {
        // ============================ copy groups ============================
        const int cg = (warp - 2) >> 2, quad = warp & 3;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        for (int li = cg; li < n_act; li += CPY_GROUPS) {
            const int s = li % STAGES, j = li % BUFS, u = li / BUFS;
            bool w = mbar_wait(&full[s], (li / STAGES) & 1, a.budget, a.st);
            if (u > 0) w = w && mbar_wait(&done[j], (u - 1) & 1, a.budget, a.st);
            if (!__all_sync(0xffffffffu, w)) break;
            tc_fence_after();
            const uint8_t* st_base = sStage + s * MX_STAGE;
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                // 68-byte rows are 17 words apart: a warp's 32 rows hit 32 banks
                const uint8_t* src = st_base + (sub * SUB + quad * 32 + lane) * MX_ROW;
                uint32_t c[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) c[i] = ld_u32(src + 4 * i);
                uint32_t sf[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) sf[q4] = ld_u32(st_base + (sub * SUB + lane + 32 * q4) * MX_ROW + CODE_BYTES);
                tmem_st16(tmem + lane_base + A_COL0 + j * 32 + sub * 16, c);
                tmem_st4(tmem + lane_base + SFA_COL0 + j * 8 + sub * 4, sf[0], sf[1], sf[2], sf[3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[j]);
        }
    } else {
        // ============================ epilogue groups ============================
        const int eg = (warp - 2 - 4 * CPY_GROUPS) >> 2, quad = warp & 3;
        const int64_t n_elems = CAND ? (int64_t)a.n_pool * 8 : a.N;
        const int64_t nb = (a.N + 7) / 8;
        const uint32_t tb0 = tmem + ((uint32_t)(quad * 32) << 16) + D_COL0;
        const float4* w4 = reinterpret_cast<const float4*>(sW);
        for (int li = eg; li < n_act; li += EPI_GROUPS) {
            const int j = li % BUFS;
            {
                const bool w = mbar_wait(&done[j], (li / BUFS) & 1, a.budget, a.st);
                if (!__all_sync(0xffffffffu, w)) break;
            }
            tc_fence_after();
            const int tile = t_begin + li;
#pragma unroll 1
            for (int sub = 0; sub < 2; ++sub) {
                const int64_t e = (int64_t)tile * TILE + sub * SUB + quad * 32 + lane;
                int64_t sid = e;
                if (CAND) {
                    const int64_t pi = e >> 3;
                    const int32_t pb = pi < a.n_pool ? a.pool[(int64_t)g * a.n_pool + pi] : -1;
                    sid = (pb >= 0 && (int64_t)pb * 8 + 8 <= a.N) ? (int64_t)pb * 8 + (e & 7) : INT64_MAX;
                }
                // four chains (head h feeds chain h mod 4) of w_h * 2 ReLU(d_h), over the
                // two 32-head halves of the sub-tile's D (32 registers at a time)
                float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t d[32];
                    tmem_ld32(tb0 + j * 128 + sub * 64 + hh * 32, d);
                    tmem_wait_ld();
                    if (sub == 1 && hh == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&dempty[j]);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 wv = w4[hh * 8 + i];
                        const float x0 = __uint_as_float(d[4 * i]), x1 = __uint_as_float(d[4 * i + 1]);
                        const float x2 = __uint_as_float(d[4 * i + 2]), x3 = __uint_as_float(d[4 * i + 3]);
                        ffma2(a4[0], a4[1], wv.x, wv.y, x0 + fabsf(x0), x1 + fabsf(x1));
                        ffma2(a4[2], a4[3], wv.z, wv.w, x2 + fabsf(x2), x3 + fabsf(x3));
                    }
                }
                const float acc = ((a4[0] + a4[1]) + (a4[2] + a4[3])) * 0.5f;
                const bool vis = sid < V && e < n_elems;
                const float sc = vis ? acc : -INFINITY;
                if (a.scores && e < n_elems) a.scores[(int64_t)g * n_elems + e] = sc;
                if (!CAND && a.bmax) {
                    float m = sc;
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    if ((lane & 7) == 0 && (e >> 3) < nb) a.bmax[(int64_t)g * nb + (e >> 3)] = m;
                }
            }
        }
        // tiles of this CTA past every visible entry: -inf outputs
        for (int tile = t_begin + n_act + eg; tile < t_end; tile += EPI_GROUPS) {
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int64_t e = (int64_t)tile * TILE + sub * SUB + quad * 32 + lane;
                if (a.scores && e < n_elems) a.scores[(int64_t)g * n_elems + e] = -INFINITY;
                if (!CAND && a.bmax && (lane & 7) == 0 && (e >> 3) < nb)
                    a.bmax[(int64_t)g * nb + (e >> 3)] = -INFINITY;
            }
        }
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
    // the first radix digit of this CTA's visible block maxima, counted once every tile
    // is done (counting them in the epilogue stalled the pipeline), into the row's
    // histogram: the maxima are read back eight at a time, all in flight together
    if (!CAND && a.hist) {
        for (int i = threadIdx.x; i < CSA2_BLOCK_HIST_BINS; i += THREADS) sHist[i] = 0u;
        __syncthreads();
        const int64_t nbv = (V + 7) / 8, b0 = (int64_t)t_begin * (TILE / 8);
        const int64_t b1 = min(nbv, (int64_t)t_end * (TILE / 8));
        const float* brow = a.bmax + (int64_t)g * ((a.N + 7) / 8);
        for (int64_t base = b0; base < b1; base += 8 * THREADS) {
            float mv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int64_t bi = base + j * THREADS + threadIdx.x;
                mv[j] = bi < b1 ? brow[bi] : -INFINITY;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (mv[j] != -INFINITY) atomicAdd(&sHist[order_key(mv[j]) >> 20], 1u);
        }
        __syncthreads();
        uint32_t* hrow = a.hist + (int64_t)g * CSA2_BLOCK_HIST_BINS;
        for (int i = threadIdx.x; i < CSA2_BLOCK_HIST_BINS; i += THREADS)
            if (const uint32_t v = sHist[i]) atomicAdd(&hrow[i], v);
    }
}

template <bool CAND>
csa2_status launch_fp4(csa2_ctx* ctx, FpArgs& a, cudaStream_t s) {
    auto kern = index_scan_fp4_kernel<CAND>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
            return CSA2_ERR_CUDA;
        attr = true;
    }
    const int groups = a.B * a.Q;
    int splits = (int)std::min<int64_t>(a.tiles, std::max<int64_t>(1, ((int64_t)ctx->num_sms + groups - 1) / groups));
    a.tiles_per_cta = (a.tiles + splits - 1) / splits;
    splits = (a.tiles + a.tiles_per_cta - 1) / a.tiles_per_cta;
    const csa2_status r = launch_pdl(kern, dim3((unsigned)splits, (unsigned)groups), dim3(THREADS), SMEM, s, a);
    return r != CSA2_OK ? r : csa2_launch_status();
}

}  // namespace

csa2_status index_score_fp4_dispatch(csa2_ctx* ctx, const void* q_idx, const float* w, const void* k_idx, int B,
                                     int Q, int64_t N, int H_I, const int64_t* n_visible, const int32_t* pool,
                                     int n_pool, int block, float* scores, float* block_max, uint32_t* hist,
                                     cudaStream_t s, const void* q_bf16, uint8_t* q_mx_out) {
    if (H_I != HEADS || block != 8 || (N % 8) != 0 || N == 0) return CSA2_ERR_UNSUPPORTED;
    if (pool && (n_pool % BLOCKS_PER_TILE) != 0) return CSA2_ERR_UNSUPPORTED;
    FpArgs a;
    a.qmx = reinterpret_cast<const uint8_t*>(q_idx);
    a.qbf = reinterpret_cast<const __nv_bfloat16*>(q_bf16);
    a.qmx_out = q_mx_out;
    a.w = w;
    a.kmx = reinterpret_cast<const uint8_t*>(k_idx);
    a.nv = n_visible;
    a.pool = pool;
    a.scores = scores;
    a.bmax = block_max;
    a.hist = pool ? nullptr : hist;
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
    a.tiles = pool ? n_pool / BLOCKS_PER_TILE : (int)((N + TILE - 1) / TILE);
    if (a.tiles == 0) return CSA2_OK;
    return pool ? launch_fp4<true>(ctx, a, s) : launch_fp4<false>(ctx, a, s);
}
