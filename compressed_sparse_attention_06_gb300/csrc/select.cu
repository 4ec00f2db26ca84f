// Deterministic top-k selection and the hierarchical block pool.
//
// Top-k (DSA-to-CSA/HCA page eq. (17)) and the pool (CSA2 page,
// «解码器里的分层索引»; Attention-evolution page §4.4) share one kernel: a CTA per
// row finds the exact k-th largest key by 4 passes of 8-bit radix histograms over
// the order-preserving uint32 of each score, then writes the winners in index order
// (one coalesced pass with block-wide scans).  Keys equal to the threshold are taken
// lowest index first, so the order is (score desc, index asc) with no dependence on
// thread timing.
#include "csa2_internal.cuh"

namespace {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;

enum SelMode { SEL_TOPK = 0, SEL_CAND = 1, SEL_POOL = 2 };

struct SelArgs {
    const float* vals;        // scores (topk / candidates) or block maxima (pool)
    int64_t n;                // elements per row (topk: N; cand: n_pool*block; pool: ld)
    int64_t ld;               // row stride of vals
    const int64_t* nv;        // visible entries per row
    const int32_t* pool;      // candidate mode: [rows, n_pool]
    int n_pool;
    int block;
    int k;                    // winners wanted (pool: n_keep - 1, newest block added after)
    int out_len;              // output row length (topk: k; pool: n_keep)
    int32_t* out_idx;
    float* out_val;
    unsigned int* st;         // context status word (out-of-range rows are flagged)
};

struct ElemInfo {
    bool valid;
    int64_t id;
};

template <int MODE>
__device__ __forceinline__ ElemInfo elem_info(const SelArgs& a, int64_t row, int64_t e, int64_t V,
                                              int64_t n_elems) {
    ElemInfo r;
    r.valid = false;
    r.id = e;
    if (e >= n_elems) return r;
    if (MODE == SEL_TOPK) {
        r.valid = e < V;
    } else if (MODE == SEL_CAND) {
        int32_t pb = a.pool[row * a.n_pool + e / a.block];
        r.id = (int64_t)pb * a.block + e % a.block;
        r.valid = pb >= 0 && r.id < V;
    } else {
        // blocks 0 .. nb-1 are visible; the newest (nb-1) is added separately
        const int64_t nb = (V + a.block - 1) / a.block;
        r.valid = e < nb - 1;
    }
    return r;
}

// Block-wide exclusive scan of a 0/1 flag; returns the prefix, writes the total.
__device__ __forceinline__ int block_excl_scan(bool flag, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned bal = __ballot_sync(0xffffffffu, flag);
    int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[wid] = __popc(bal);
    __syncthreads();
    if (wid == 0) {
        int v = warp_tot[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        warp_tot[lane] = incl - v;              // exclusive
        if (lane == 31) warp_tot[32] = incl;    // total
    }
    __syncthreads();
    int r = warp_tot[wid] + in_warp;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

template <int MODE>
__global__ void __launch_bounds__(SEL_THREADS) select_kernel(SelArgs a) {
    __shared__ unsigned int hist[256];
    __shared__ int warp_tot[33];
    __shared__ unsigned int s_digit;
    __shared__ int s_remaining;
    __shared__ unsigned int s_nvalid;

    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t V = a.nv[row];
    const float* vals = a.vals + row * a.ld;
    int64_t n_elems = (MODE == SEL_POOL) ? (V > 0 ? ((V + a.block - 1) / a.block) : 0) : a.n;
    if (MODE == SEL_POOL && n_elems > a.ld) {
        // more visible blocks than the row holds: flag it and use what is there
        if (tid == 0) csa2_flag(a.st, CSA2_DEVBIT_RANGE);
        n_elems = a.ld;
    }
    const int k = a.k;

    uint32_t prefix = 0, pmask = 0;
    int remaining = k;
    bool take_all = false;
    for (int pass = 0; pass < 4 && k > 0; ++pass) {
        const int shift = 24 - 8 * pass;
        if (tid < 256) hist[tid] = 0;
        if (tid == 0) s_nvalid = 0;
        __syncthreads();
        unsigned int local_valid = 0;
        for (int64_t e = tid; e < n_elems; e += SEL_THREADS) {
            ElemInfo inf = elem_info<MODE>(a, row, e, V, n_elems);
            if (!inf.valid) continue;
            ++local_valid;
            uint32_t key = order_key(vals[e]);
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        if (pass == 0) {
            local_valid = __reduce_add_sync(0xffffffffu, local_valid);
            if ((tid & 31) == 0 && local_valid) atomicAdd(&s_nvalid, local_valid);
        }
        __syncthreads();
        if (pass == 0 && s_nvalid <= (unsigned)k) {
            take_all = true;
            break;
        }
        if (tid < 32) {
            const int lane = tid;
            unsigned int loc[8];
            unsigned int lsum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                loc[j] = hist[255 - 8 * lane - j];
                lsum += loc[j];
            }
            unsigned int incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            unsigned int excl = incl - lsum;
            if (excl < (unsigned)remaining && (unsigned)remaining <= incl) {
                unsigned int cum = excl;
                for (int j = 0; j < 8; ++j) {
                    if (cum + loc[j] >= (unsigned)remaining) {
                        s_digit = 255u - 8u * lane - j;
                        s_remaining = remaining - (int)cum;
                        break;
                    }
                    cum += loc[j];
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= 255u << shift;
        remaining = s_remaining;
        __syncthreads();
    }
    const uint32_t T = prefix;

    // ordered compaction: winners are keys > T, plus the first `remaining` keys == T
    int eq_run = 0, out_run = 0;
    for (int64_t base = 0; base < n_elems && out_run < k; base += SEL_THREADS) {
        const int64_t e = base + tid;
        ElemInfo inf = elem_info<MODE>(a, row, e, V, n_elems);
        float v = inf.valid ? vals[e] : 0.0f;
        uint32_t key = inf.valid ? order_key(v) : 0u;
        bool gt, eq;
        if (take_all) {
            gt = inf.valid;
            eq = false;
        } else {
            gt = inf.valid && key > T;
            eq = inf.valid && key == T;
        }
        int eq_tot;
        int eq_rank = block_excl_scan(eq, warp_tot, eq_tot) + eq_run;
        bool sel = gt || (eq && eq_rank < remaining);
        int sel_tot;
        int pos = block_excl_scan(sel, warp_tot, sel_tot) + out_run;
        if (sel && pos < k) {
            a.out_idx[row * a.out_len + pos] = (int32_t)inf.id;
            if (a.out_val) a.out_val[row * a.out_len + pos] = v;
        }
        eq_run += eq_tot;
        out_run += sel_tot;
    }
    if (out_run > k) out_run = k;
    int filled = out_run;
    if (MODE == SEL_POOL && n_elems > 0) {
        // the newest visible block is always kept; it is the largest id
        if (tid == 0) a.out_idx[row * a.out_len + filled] = (int32_t)(n_elems - 1);
        ++filled;
    }
    for (int i = filled + tid; i < a.out_len; i += SEL_THREADS) {
        a.out_idx[row * a.out_len + i] = -1;
        if (a.out_val) a.out_val[row * a.out_len + i] = -INFINITY;
    }
}

}  // namespace

extern "C" csa2_status csa2_topk(csa2_ctx* ctx, const float* scores, int64_t rows, int64_t n, int64_t ld,
                                 const int64_t* n_visible, const int32_t* pool_blocks, int n_pool, int block,
                                 int k, int32_t* out_idx, float* out_score, void* stream) {
    if (!ctx || rows < 0 || n < 0 || k < 1 || k > 4096) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (rows > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED;
    if (!scores || !n_visible || !out_idx) return CSA2_ERR_INVALID_ARG;
    SelArgs a;
    a.vals = scores;
    a.ld = ld;
    a.nv = n_visible;
    a.pool = pool_blocks;
    a.n_pool = n_pool;
    a.block = block;
    a.k = k;
    a.out_len = k;
    a.out_idx = out_idx;
    a.out_val = out_score;
    a.st = ctx->status;
    cudaStream_t s = as_stream(stream);
    if (pool_blocks) {
        if (block < 1 || n_pool < 0) return CSA2_ERR_INVALID_ARG;
        a.n = (int64_t)n_pool * block;
        if (ld < a.n) return CSA2_ERR_INVALID_ARG;
        select_kernel<SEL_CAND><<<(unsigned)rows, SEL_THREADS, 0, s>>>(a);
    } else {
        if (ld < n) return CSA2_ERR_INVALID_ARG;
        a.n = n;
        select_kernel<SEL_TOPK><<<(unsigned)rows, SEL_THREADS, 0, s>>>(a);
    }
    return csa2_launch_status();
}

extern "C" csa2_status csa2_block_pool(csa2_ctx* ctx, const float* block_max, int64_t rows, int64_t ld,
                                       const int64_t* n_visible, int block, int n_keep, int32_t* out_blocks,
                                       void* stream) {
    if (!ctx || rows < 0 || ld < 0 || block < 1 || n_keep < 1 || n_keep > 4096) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (rows > 0x7FFFFFFF) return CSA2_ERR_UNSUPPORTED;
    if (!block_max || !n_visible || !out_blocks) return CSA2_ERR_INVALID_ARG;
    SelArgs a;
    a.vals = block_max;
    a.n = ld;
    a.ld = ld;
    a.nv = n_visible;
    a.pool = nullptr;
    a.n_pool = 0;
    a.block = block;
    a.k = n_keep - 1;
    a.out_len = n_keep;
    a.out_idx = out_blocks;
    a.out_val = nullptr;
    a.st = ctx->status;
    select_kernel<SEL_POOL><<<(unsigned)rows, SEL_THREADS, 0, as_stream(stream)>>>(a);
    return csa2_launch_status();
}
