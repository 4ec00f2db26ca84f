// Deterministic top-k selection and the hierarchical block pool.
//
// Top-k (DSA-to-CSA/HCA page eq. (17)) and the pool (CSA2 page,
// «解码器里的分层索引»; Attention-evolution page §4.4) share one exact radix select:
// every score becomes an order-preserving uint32 key, a 12-bit histogram and two
// 10-bit histograms (the last two over the keys of the threshold bin only) find the
// k-th largest key T, and one ordered pass emits the keys above T plus the first
// (lowest-index) keys equal to T.  The result is the top-k in the order
// (score desc, index asc), independent of thread timing.
//
// Layouts:
//   * a row that fits (<= SEL_SMEM_CAP elements) is staged in shared memory once and
//     every pass runs there, one CTA per row;
//   * a long row with few rows (the 1M-context pool: 131,072 blocks per query) is
//     split over several CTAs; each keeps its chunk's top-k (key, id) pairs in the
//     caller's workspace, and a merge CTA per row selects the final top-k from
//     those (the union of per-chunk top-k lists contains the row's top-k under the
//     same total order);
//   * without a workspace a long row falls back to one CTA reading global memory
//     on every pass;
//   * few long rows (decode) run as one thread-block cluster per row, the digits
//     counted per CTA and combined through distributed shared memory (cluster
//     selection, below);
//   * the decode pool, and the pool fused with the top-k of the best blocks' entries
//     (csa2_pool_topk), start from the first-digit histogram the indexer scan counted
//     (pool from a histogram, below).
// The threshold search takes a 12-bit histogram over every key, copies the keys of
// the threshold bin aside and resolves the remaining 20 bits on that copy; a warp
// whose keys share a digit (scores of one row often share their top bits) counts
// them with one shared-memory atomic.
#include <algorithm>

#include "csa2_internal.cuh"
#include "index_score_tc.cuh"

namespace {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_SMEM_CAP = 40960;        // keys staged in shared memory (160 KB)

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
    int chunks;               // > 1: two-stage path through the workspace
    int64_t chunk_len;
    uint32_t* ws_key;         // [rows, chunks, k]
    int32_t* ws_id;           // [rows, chunks, k]
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
        const int32_t pb = a.pool[row * a.n_pool + e / a.block];
        r.id = (int64_t)pb * a.block + e % a.block;
        r.valid = pb >= 0 && r.id < V;
    } else {
        r.valid = e < n_elems - 1;          // the newest visible block is added separately
    }
    return r;
}

// Elements of a row: candidate / score count, or the visible blocks for the pool.
template <int MODE>
__device__ __forceinline__ int64_t row_elems(const SelArgs& a, int64_t V) {
    if (MODE != SEL_POOL) return a.n;
    int64_t nb = V > 0 ? (V + a.block - 1) / a.block : 0;
    if (nb > a.ld) {
        if (threadIdx.x == 0 && blockIdx.x == 0) csa2_flag(a.st, CSA2_DEVBIT_RANGE);
        nb = a.ld;
    }
    return nb;
}

// Key of a valid score: order-preserving, never 0 (0 marks "not a candidate"; only an
// all-ones NaN would map to 0 and NaN scores are outside the contract).
template <int MODE>
__device__ __forceinline__ uint32_t key_of(const SelArgs& a, int64_t row, int64_t e, int64_t V, int64_t n_elems) {
    ElemInfo inf = elem_info<MODE>(a, row, e, V, n_elems);
    return inf.valid ? order_key(a.vals[row * a.ld + e]) : 0u;
}

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr int NB_A = 4096;             // first digit: key bits 31..20
constexpr int NB_B = 1024;             // then bits 19..10 and 9..0
constexpr int CAND_CAP = 8192;         // keys of the threshold bin kept for the last two digits

struct SelState {
    uint32_t T;
    int remaining;
    bool take_all;
};

struct SelShared {
    uint32_t hist[NB_A];
    uint32_t wtot[32];
    uint32_t wtot_all;
    int warp_tot[33];
    int bin, nvalid, cand_n;
    uint32_t above;
};

// Block-wide exclusive scan of one value per thread (thread order); `total` gets the sum.
template <class Sh>
__device__ __forceinline__ uint32_t block_excl_scan_u32(uint32_t v, Sh& sh, uint32_t& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) sh.wtot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const uint32_t t = lane < nw ? sh.wtot[lane] : 0u;
        uint32_t ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(FULL_MASK, ti, o);
            if (lane >= o) ti += u;
        }
        sh.wtot[lane] = ti - t;
        if (lane == 31) sh.wtot_all = ti;
    }
    __syncthreads();
    const uint32_t r = sh.wtot[wid] + incl - v;
    total = sh.wtot_all;
    __syncthreads();
    return r;
}

// Count digit d of every active lane: a warp whose active lanes share one digit adds
// once; otherwise each active lane adds its own (shared-memory atomics).
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t d, bool act) {
    const unsigned am = __ballot_sync(FULL_MASK, act);
    if (am == 0u) return;
    const int leader = __ffs(am) - 1;
    const uint32_t d0 = __shfl_sync(FULL_MASK, d, leader);
    if (__all_sync(FULL_MASK, !act || d == d0)) {
        if ((int)(threadIdx.x & 31) == leader) atomicAdd(&hist[d0], (uint32_t)__popc(am));
    } else if (act) {
        atomicAdd(&hist[d], 1u);
    }
}

// Histogram of digit (key >> shift) & dmask over the active keys (valid, and equal to
// `prefix` on the bits of `pmask`).
template <class KeyAt>
__device__ __forceinline__ void hist_pass(KeyAt key_at, int64_t n, uint32_t prefix, uint32_t pmask, int shift,
                                          uint32_t dmask, uint32_t* hist, int* nvalid) {
    const int lane = threadIdx.x & 31;
    int local_valid = 0;
    for (int64_t base = 0; base < n; base += blockDim.x) {
        const int64_t e = base + threadIdx.x;
        const uint32_t key = e < n ? key_at(e) : 0u;
        local_valid += key != 0u;
        const bool act = key != 0u && (key & pmask) == prefix;
        hist_add_warp(hist, (key >> shift) & dmask, act);
    }
    if (nvalid) {
        const int w = __reduce_add_sync(FULL_MASK, local_valid);
        if (lane == 0 && w) atomicAdd(nvalid, w);
    }
}

// The bin (searched from the top) that holds the `remaining`-th largest active key:
// sh.bin = that bin, sh.above = active keys in the bins above it.  nb is a multiple
// of the block size.
template <class Sh>
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, uint32_t remaining, Sh& sh) {
    const int per = nb / (int)blockDim.x;
    const int top = nb - 1 - (int)threadIdx.x * per;
    uint32_t loc = 0;
    for (int j = 0; j < per; ++j) loc += hist[top - j];
    uint32_t total;
    const uint32_t excl = block_excl_scan_u32(loc, sh, total);
    if (excl < remaining && remaining <= excl + loc) {
        uint32_t cum = excl;
        for (int j = 0; j < per; ++j) {
            const uint32_t c = hist[top - j];
            if (cum + c >= remaining) {
                sh.bin = top - j;
                sh.above = cum;
                break;
            }
            cum += c;
        }
    }
    __syncthreads();
}

// Unordered copy of the active keys into cand (sh.cand_n must start at 0).
template <class KeyAt>
__device__ __forceinline__ void compact_active(KeyAt key_at, int64_t n, uint32_t prefix, uint32_t pmask,
                                               uint32_t* cand, SelShared& sh) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t base = 0; base < n; base += blockDim.x) {
        const int64_t e = base + threadIdx.x;
        const uint32_t key = e < n ? key_at(e) : 0u;
        const bool act = key != 0u && (key & pmask) == prefix;
        const unsigned am = __ballot_sync(FULL_MASK, act);
        if (am == 0u) continue;
        const int leader = __ffs(am) - 1;
        int off = 0;
        if (lane == leader) off = atomicAdd(&sh.cand_n, __popc(am));
        off = __shfl_sync(FULL_MASK, off, leader);
        if (act) cand[off + __popc(am & lt)] = key;
    }
}

// Exact k-th largest key over n elements given by key_at(e) (0 = not a candidate):
// a 12-bit histogram over all keys picks the threshold bin; its keys (if at most
// CAND_CAP) are copied aside and two 10-bit passes over them finish the key.
template <class KeyAt>
__device__ SelState block_radix_select(KeyAt key_at, int64_t n, int k, SelShared& sh, uint32_t* cand) {
    const int tid = threadIdx.x;
    SelState r;
    r.take_all = false;
    r.T = 0xFFFFFFFFu;
    r.remaining = 0;
    if (k <= 0) return r;
    for (int i = tid; i < NB_A; i += blockDim.x) sh.hist[i] = 0;
    if (tid == 0) {
        sh.nvalid = 0;
        sh.cand_n = 0;
    }
    __syncthreads();
    hist_pass(key_at, n, 0u, 0u, 20, 0xFFFu, sh.hist, &sh.nvalid);
    __syncthreads();
    if (sh.nvalid <= k) {
        r.take_all = true;
        r.T = 0;
        return r;
    }
    find_bin(sh.hist, NB_A, (uint32_t)k, sh);
    uint32_t prefix = (uint32_t)sh.bin << 20, pmask = 0xFFF00000u;
    uint32_t remaining = (uint32_t)k - sh.above;
    const uint32_t m = sh.hist[sh.bin];
    __syncthreads();
    const bool use_cand = m <= (uint32_t)CAND_CAP;
    if (use_cand) {
        compact_active(key_at, n, prefix, pmask, cand, sh);
        __syncthreads();
    }
    auto cand_at = [&](int64_t i) -> uint32_t { return cand[i]; };
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        for (int i = tid; i < NB_B; i += blockDim.x) sh.hist[i] = 0;
        __syncthreads();
        if (use_cand)
            hist_pass(cand_at, (int64_t)m, prefix, pmask, shift, 0x3FFu, sh.hist, nullptr);
        else
            hist_pass(key_at, n, prefix, pmask, shift, 0x3FFu, sh.hist, nullptr);
        __syncthreads();
        find_bin(sh.hist, NB_B, remaining, sh);
        prefix |= (uint32_t)sh.bin << shift;
        pmask |= 0x3FFu << shift;
        remaining -= sh.above;
        __syncthreads();
    }
    r.T = prefix;
    r.remaining = (int)remaining;
    return r;
}

// Emit the winners in element order: keys > T, then the first `remaining` keys == T.
// Each warp owns one contiguous segment: it counts its winners, one prefix over the
// warp totals gives every warp its output offset and its rank among the ties, and
// each warp then writes its winners in order (ballot prefix sums, two barriers).
template <class KeyAt, class Emit>
__device__ int block_ordered_emit(KeyAt key_at, int64_t n, const SelState& r, int k, SelShared& sh, Emit emit) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const int64_t seg = ((n + nw - 1) / nw + 31) / 32 * 32;
    const int64_t s0 = (int64_t)wid * seg, s1 = min(n, s0 + seg);
    int cnt_gt = 0, cnt_eq = 0;
    for (int64_t base = s0; base < s1; base += 32) {
        const int64_t e = base + lane;
        const uint32_t key = e < s1 ? key_at(e) : 0u;
        const bool valid = key != 0u;
        const bool gt = r.take_all ? valid : (valid && key > r.T);
        const bool eq = !r.take_all && valid && key == r.T;
        cnt_gt += __popc(__ballot_sync(0xffffffffu, gt));
        cnt_eq += __popc(__ballot_sync(0xffffffffu, eq));
    }
    int* wgt = sh.warp_tot;            // [32] gt counts, then exclusive prefixes
    __shared__ int weq[32];
    if (lane == 0) {
        wgt[wid] = cnt_gt;
        weq[wid] = cnt_eq;
    }
    __syncthreads();
    if (wid == 0) {
        const int g = lane < nw ? wgt[lane] : 0, q = lane < nw ? weq[lane] : 0;
        int ig = g, iq = q;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ug = __shfl_up_sync(0xffffffffu, ig, o), uq = __shfl_up_sync(0xffffffffu, iq, o);
            if (lane >= o) {
                ig += ug;
                iq += uq;
            }
        }
        if (lane < nw) {
            wgt[lane] = ig - g;        // gt before this warp
            weq[lane] = iq - q;        // ties before this warp
        }
        if (lane == 31) sh.warp_tot[32] = ig + min(iq, r.remaining);
    }
    __syncthreads();
    const int gt_before = wgt[wid], eq_before = weq[wid];
    int run_gt = 0, run_eq = 0;
    for (int64_t base = s0; base < s1; base += 32) {
        const int64_t e = base + lane;
        const uint32_t key = e < s1 ? key_at(e) : 0u;
        const bool valid = key != 0u;
        const bool gt = r.take_all ? valid : (valid && key > r.T);
        const bool eq = !r.take_all && valid && key == r.T;
        const unsigned bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
        const int eq_rank = eq_before + run_eq + __popc(be & lt);
        const bool tie_in = eq && eq_rank < r.remaining;
        const int sel_eq_before = min(eq_before + run_eq, r.remaining);
        const unsigned bs = __ballot_sync(0xffffffffu, tie_in);
        const int pos = gt_before + run_gt + sel_eq_before + __popc(bg & lt) + __popc(bs & lt);
        if ((gt || tie_in) && pos < k) emit(e, pos, key);
        run_gt += __popc(bg);
        run_eq += __popc(be);
    }
    const int total = sh.warp_tot[32];
    __syncthreads();
    return min(total, k);
}

constexpr int BM_WORDS = SEL_SMEM_CAP / 32;     // bitmap words for a staged row

// Keys staged in shared memory (zero-padded to whole words of 32).
struct SmemKeys {
    const uint32_t* skey;
    __device__ __forceinline__ uint4 piece(int w, int q) const {
        return reinterpret_cast<const uint4*>(skey)[w * 8 + q];
    }
    __device__ __forceinline__ uint32_t key(int i) const { return skey[i]; }
};

// Keys computed on the fly from one row of scores in global memory (16-byte
// aligned): element i < V (and < n) is visible.
struct RowScores {
    const float* rowp;
    int n, V;
    __device__ __forceinline__ uint32_t key(int i) const { return (i < V && i < n) ? order_key(rowp[i]) : 0u; }
    __device__ __forceinline__ uint4 piece(int w, int q) const {
        const int e = 32 * w + 4 * q;
        const int lim = min(n, V);
        if (e + 3 < lim) {
            const float4 f = reinterpret_cast<const float4*>(rowp)[e >> 2];
            return make_uint4(order_key(f.x), order_key(f.y), order_key(f.z), order_key(f.w));
        }
        return make_uint4(key(e), key(e + 1), key(e + 2), key(e + 3));
    }
};
constexpr int CAND64_CAP = CAND_CAP / 2;        // (key, index) pairs in the candidate buffer

// Selection over keys staged in shared memory, whose 12-bit histogram (sh.hist) and
// valid count were built while staging and exceed k.  The threshold bin b is found
// from the histogram; keys above b are winners outright, the keys of b (at most
// CAND64_CAP) are copied with their index and two 10-bit histograms over the copy
// give the exact threshold key T and how many ties at T are taken.  Winners and ties
// are marked in two bitmaps (bmW, bmE: zeroed by the caller), and one ordered scan of
// the bitmaps emits the winners in element order, the lowest-index ties first.
// Returns -1 (nothing emitted) if bin b holds more than CAND64_CAP keys.
template <class Src, class Emit>
__device__ int staged_select(const Src src, int n, int k, SelShared& sh, uint64_t* cand, uint32_t* bmW,
                             uint32_t* bmE, Emit emit) {
    const int tid = threadIdx.x;
    find_bin(sh.hist, NB_A, (uint32_t)k, sh);
    const uint32_t b = (uint32_t)sh.bin;
    uint32_t remaining = (uint32_t)k - sh.above;
    const uint32_t m = sh.hist[b];
    if (tid == 0) sh.cand_n = 0;
    __syncthreads();
    if (m > (uint32_t)CAND64_CAP) return -1;
    // classify: a thread per word of 32 keys (bit j of word w = key 32w + j), read as
    // eight 16-byte pieces starting at a lane-dependent piece so that the lanes of a
    // warp spread over the banks; skey is padded with zeros to a whole word
    const int nwords = (n + 31) / 32;
    const int lane = tid & 31;
    for (int w0 = 0; w0 < nwords; w0 += blockDim.x) {
        const int w = w0 + tid;
        uint32_t mgt = 0u, meq = 0u;
        if (w < nwords) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int q = (t + w) & 7;
                const uint4 k4 = src.piece(w, q);
                const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t key = kk[c], d = key >> 20;
                    if (key != 0u && d > b) mgt |= 1u << (4 * q + c);
                    if (key != 0u && d == b) meq |= 1u << (4 * q + c);
                }
            }
            bmW[w] = mgt;
        }
        // the bin's keys go to cand: one atomic per warp, offsets by a warp scan
        const int cnt = __popc(meq);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += u;
        }
        int base = 0;
        if (lane == 31 && incl) base = atomicAdd(&sh.cand_n, incl);
        base = __shfl_sync(FULL_MASK, base, 31) + incl - cnt;
        while (meq) {
            const int j = __ffs(meq) - 1;
            meq &= meq - 1;
            cand[base++] = ((uint64_t)src.key(w * 32 + j) << 32) | (uint32_t)(w * 32 + j);
        }
    }
    __syncthreads();
    // the low 20 bits of T among the bin's keys
    auto cand_key = [&](int64_t j) -> uint32_t { return (uint32_t)(cand[j] >> 32); };
    uint32_t prefix = b << 20, pmask = 0xFFF00000u;
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        for (int i = tid; i < NB_B; i += blockDim.x) sh.hist[i] = 0;
        __syncthreads();
        hist_pass(cand_key, (int64_t)m, prefix, pmask, shift, 0x3FFu, sh.hist, nullptr);
        __syncthreads();
        find_bin(sh.hist, NB_B, remaining, sh);
        prefix |= (uint32_t)sh.bin << shift;
        pmask |= 0x3FFu << shift;
        remaining -= sh.above;
        __syncthreads();
    }
    const uint32_t T = prefix;
    for (int j = tid; j < (int)m; j += blockDim.x) {
        const uint64_t c = cand[j];
        const uint32_t key = (uint32_t)(c >> 32), i = (uint32_t)c;
        if (key > T) atomicOr(&bmW[i >> 5], 1u << (i & 31));
        else if (key == T) atomicOr(&bmE[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    // ordered emission: thread t owns a run of consecutive words
    const int per = (nwords + (int)blockDim.x - 1) / (int)blockDim.x;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    uint32_t cg = 0, ce = 0;
    for (int w = w0; w < w1; ++w) {
        cg += __popc(bmW[w]);
        ce += __popc(bmE[w]);
    }
    // both counts in one scan: a chunk holds fewer than 2^16 keys, so neither half carries
    uint32_t tot;
    const uint32_t both = block_excl_scan_u32(cg | (ce << 16), sh, tot);
    uint32_t gb = both & 0xFFFFu, eb = both >> 16;
    for (int w = w0; w < w1; ++w) {
        const uint32_t wg = bmW[w], we = bmE[w];
        uint32_t bits = wg | we;
        while (bits) {
            const int j = __ffs(bits) - 1;
            bits &= bits - 1;
            const int i = w * 32 + j;
            if ((wg >> j) & 1u) {
                emit((int64_t)i, (int)(gb + min(eb, remaining)), src.key(i));
                ++gb;
            } else {
                if (eb < remaining) emit((int64_t)i, (int)(gb + eb), src.key(i));
                ++eb;
            }
        }
    }
    __syncthreads();
    return k;
}

// Stage n keys from load(i) into skey while building their 12-bit histogram and
// valid count (eight loads in flight per thread); also zeroes the bitmaps.
template <class Load>
__device__ void stage_keys(Load load, int n, uint32_t* skey, SelShared& sh, uint32_t* bmW, uint32_t* bmE) {
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < NB_A; i += blockDim.x) sh.hist[i] = 0;
    for (int i = tid; i < (n + 31) / 32; i += blockDim.x) {
        bmW[i] = 0u;
        bmE[i] = 0u;
    }
    if (tid == 0) {
        sh.nvalid = 0;
        sh.cand_n = 0;
    }
    __syncthreads();
    int local_valid = 0;
    for (int base = 0; base < n; base += (int)blockDim.x * 8) {
        uint32_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = base + j * (int)blockDim.x + tid;
            v[j] = i < n ? load(i) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = base + j * (int)blockDim.x + tid;
            if (i < n) skey[i] = v[j];
            local_valid += v[j] != 0u;
            hist_add_warp(sh.hist, v[j] >> 20, v[j] != 0u);
        }
    }
    for (int i = n + tid; i < (n + 31) / 32 * 32; i += blockDim.x) skey[i] = 0u;
    const int w = __reduce_add_sync(FULL_MASK, local_valid);
    if (lane == 0 && w) atomicAdd(&sh.nvalid, w);
    __syncthreads();
}

// Full-row top-k staging: scores[0..n) of one row, visible below V, into skey as keys,
// with their 12-bit histogram and valid count (16-byte loads and stores when the row
// is 16-byte aligned; spread scores, so the histogram takes plain atomics).
__device__ void stage_scores(const float* rowp, int n, int V, uint32_t* skey, SelShared& sh, uint32_t* bmW,
                             uint32_t* bmE) {
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < NB_A; i += blockDim.x) sh.hist[i] = 0;
    for (int i = tid; i < (n + 31) / 32; i += blockDim.x) {
        bmW[i] = 0u;
        bmE[i] = 0u;
    }
    if (tid == 0) {
        sh.nvalid = 0;
        sh.cand_n = 0;
    }
    __syncthreads();
    int local_valid = 0;
    const bool vec = (reinterpret_cast<uintptr_t>(rowp) & 15u) == 0;
    const int nq = vec ? n / 4 : 0;
    for (int base = 0; base < nq; base += (int)blockDim.x * 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = base + j * (int)blockDim.x + tid;
            v[j] = q < nq ? reinterpret_cast<const float4*>(rowp)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = base + j * (int)blockDim.x + tid;
            if (q >= nq) continue;
            const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t kk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                kk[c] = (4 * q + c < V) ? order_key(f[c]) : 0u;
                if (kk[c]) {
                    ++local_valid;
                    atomicAdd(&sh.hist[kk[c] >> 20], 1u);
                }
            }
            if (skey) reinterpret_cast<uint4*>(skey)[q] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
        }
    }
    for (int i = 4 * nq + tid; i < n; i += blockDim.x) {
        const uint32_t key = i < V ? order_key(rowp[i]) : 0u;
        if (skey) skey[i] = key;
        if (key) {
            ++local_valid;
            atomicAdd(&sh.hist[key >> 20], 1u);
        }
    }
    if (skey)
        for (int i = n + tid; i < (n + 31) / 32 * 32; i += blockDim.x) skey[i] = 0u;
    const int w = __reduce_add_sync(FULL_MASK, local_valid);
    if (lane == 0 && w) atomicAdd(&sh.nvalid, w);
    __syncthreads();
}

// Staged keys -> winners in element order through emit(i, pos, key); returns the
// number emitted (min(valid, k)).
template <class Emit>
__device__ int select_staged_row(const uint32_t* skey, int n, int k, SelShared& sh, uint32_t* cand32,
                                 uint32_t* bmW, uint32_t* bmE, Emit emit) {
    auto key_at = [&](int64_t i) -> uint32_t { return skey[i]; };
    if (sh.nvalid <= k) {
        SelState r;
        r.T = 0;
        r.remaining = 0;
        r.take_all = true;
        return block_ordered_emit(key_at, (int64_t)n, r, k, sh, emit);
    }
    SmemKeys src;
    src.skey = skey;
    const int f = staged_select(src, n, k, sh, reinterpret_cast<uint64_t*>(cand32), bmW, bmE, emit);
    if (f >= 0) return f;
    const SelState r = block_radix_select(key_at, (int64_t)n, k, sh, cand32);
    return block_ordered_emit(key_at, (int64_t)n, r, k, sh, emit);
}

template <int MODE>
__device__ void finish_row(const SelArgs& a, int64_t row, int filled, int64_t n_elems) {
    if (MODE == SEL_POOL && n_elems > 0) {
        if (threadIdx.x == 0) a.out_idx[row * a.out_len + filled] = (int32_t)(n_elems - 1);
        ++filled;
    }
    for (int i = filled + threadIdx.x; i < a.out_len; i += blockDim.x) {
        a.out_idx[row * a.out_len + i] = -1;
        if (a.out_val) a.out_val[row * a.out_len + i] = -INFINITY;
    }
}

// Stage 1 (or the whole selection when chunks == 1): a CTA per (chunk, row).
template <int MODE, bool SMEM>
__global__ void __launch_bounds__(SEL_THREADS) sel_chunk_kernel(SelArgs a) {
    extern __shared__ uint32_t skey[];     // [chunk_len] keys (SMEM) then [CAND_CAP] candidates
    __shared__ SelShared sh;
    const int64_t row = blockIdx.y;
    const int chunk = blockIdx.x;
    const int64_t V = a.nv[row];
    const int64_t n_elems = row_elems<MODE>(a, V);
    const int64_t c0 = (int64_t)chunk * a.chunk_len;
    const int64_t c1 = min(n_elems, c0 + a.chunk_len);
    const int64_t n = max((int64_t)0, c1 - c0);
    if (SMEM) {
        __shared__ uint32_t bmW[BM_WORDS], bmE[BM_WORDS];
        uint32_t* cand = skey + (a.chunk_len + 31) / 32 * 32;
        if (MODE == SEL_TOPK)
            stage_scores(a.vals + row * a.ld + c0, (int)n, (int)max((int64_t)0, min(V, n_elems) - c0), skey, sh, bmW,
                         bmE);
        else
            stage_keys([&](int i) -> uint32_t { return key_of<MODE>(a, row, c0 + i, V, n_elems); }, (int)n, skey,
                       sh, bmW, bmE);
        if (a.chunks > 1) {
            const int64_t base = (row * a.chunks + chunk) * (int64_t)a.k;
            const int filled = select_staged_row(skey, (int)n, a.k, sh, cand, bmW, bmE,
                                                 [&](int64_t i, int pos, uint32_t key) {
                a.ws_key[base + pos] = key;
                a.ws_id[base + pos] = (int32_t)elem_info<MODE>(a, row, c0 + i, V, n_elems).id;
            });
            for (int i = filled + threadIdx.x; i < a.k; i += blockDim.x) a.ws_key[base + i] = 0u;
            return;
        }
        const int filled = select_staged_row(skey, (int)n, a.k, sh, cand, bmW, bmE,
                                             [&](int64_t i, int pos, uint32_t key) {
            a.out_idx[row * a.out_len + pos] = (int32_t)elem_info<MODE>(a, row, c0 + i, V, n_elems).id;
            if (a.out_val) a.out_val[row * a.out_len + pos] = a.vals[row * a.ld + c0 + i];
        });
        finish_row<MODE>(a, row, filled, n_elems);
        return;
    }
    // long row without a workspace: every pass reads global memory
    auto key_at = [&](int64_t i) -> uint32_t { return key_of<MODE>(a, row, c0 + i, V, n_elems); };
    uint32_t* cand = skey;
    const SelState r = block_radix_select(key_at, n, a.k, sh, cand);
    const int filled = block_ordered_emit(key_at, n, r, a.k, sh, [&](int64_t i, int pos, uint32_t key) {
        a.out_idx[row * a.out_len + pos] = (int32_t)elem_info<MODE>(a, row, c0 + i, V, n_elems).id;
        if (a.out_val) a.out_val[row * a.out_len + pos] = a.vals[row * a.ld + c0 + i];
    });
    finish_row<MODE>(a, row, filled, n_elems);
}

// Stage 2: a CTA per row selects the top-k of its chunks' winners (in chunk order,
// which is index order).
template <int MODE>
__global__ void __launch_bounds__(SEL_THREADS) sel_merge_kernel(SelArgs a) {
    extern __shared__ uint32_t skey[];
    __shared__ SelShared sh;
    const int64_t row = blockIdx.x;
    const int64_t V = a.nv[row];
    const int64_t n_elems = row_elems<MODE>(a, V);
    const int n = a.chunks * a.k;
    const int64_t base = row * (int64_t)n;
    __shared__ uint32_t bmW[BM_WORDS], bmE[BM_WORDS];
    uint32_t* cand = skey + (n + 31) / 32 * 32;
    stage_keys([&](int i) -> uint32_t { return a.ws_key[base + i]; }, n, skey, sh, bmW, bmE);
    const int filled = select_staged_row(skey, n, a.k, sh, cand, bmW, bmE, [&](int64_t i, int pos, uint32_t key) {
        a.out_idx[row * a.out_len + pos] = a.ws_id[base + i];
        if (a.out_val) a.out_val[row * a.out_len + pos] = key_to_float(key);
    });
    finish_row<MODE>(a, row, filled, n_elems);
}

// Full-row top-k for many rows of at most SEL_SMEM_CAP scores each (prefill): a
// 512-thread CTA per row with no staged copy of the row, so two CTAs share an SM and
// overlap their phases.  The histogram pass and the classify pass both read the
// row's scores (the second read is served by L2).
constexpr int STREAM_THREADS = 512;

__global__ void __launch_bounds__(STREAM_THREADS, 2) sel_stream_kernel(SelArgs a) {
    extern __shared__ uint32_t cand32[];          // [CAND_CAP]
    __shared__ SelShared sh;
    __shared__ uint32_t bmW[BM_WORDS], bmE[BM_WORDS];
    const int64_t row = blockIdx.x;
    const int n = (int)a.n;
    const int V = (int)min((int64_t)n, max((int64_t)0, a.nv[row]));
    RowScores src;
    src.rowp = a.vals + row * a.ld;
    src.n = n;
    src.V = V;
    stage_scores(src.rowp, n, V, nullptr, sh, bmW, bmE);
    auto emit = [&](int64_t i, int pos, uint32_t key) {
        a.out_idx[row * a.out_len + pos] = (int32_t)i;
        if (a.out_val) a.out_val[row * a.out_len + pos] = src.rowp[i];
    };
    auto key_at = [&](int64_t i) -> uint32_t { return src.key((int)i); };
    int filled;
    if (sh.nvalid <= a.k) {
        SelState r;
        r.T = 0;
        r.remaining = 0;
        r.take_all = true;
        filled = block_ordered_emit(key_at, (int64_t)n, r, a.k, sh, emit);
    } else {
        filled = staged_select(src, n, a.k, sh, reinterpret_cast<uint64_t*>(cand32), bmW, bmE, emit);
        if (filled < 0) {
            const SelState r = block_radix_select(key_at, (int64_t)n, a.k, sh, cand32);
            filled = block_ordered_emit(key_at, (int64_t)n, r, a.k, sh, emit);
        }
    }
    finish_row<SEL_TOPK>(a, row, filled, n);
}

// Chunking: enough CTAs for the GPU when rows are few, each chunk holding at least 4k
// elements, chunks that fit shared memory, and a merge that fits shared memory.
void choose_chunks(const csa2_ctx* ctx, int64_t rows, int64_t n_max, int k, size_t ws_bytes, bool have_ws,
                   int& chunks, int64_t& chunk_len, bool& smem) {
    // a row that fits on-chip is one CTA: its two passes cost less than a second launch
    if (n_max <= SEL_SMEM_CAP) {
        chunks = 1;
        chunk_len = std::max<int64_t>(n_max, 1);
        smem = true;
        return;
    }
    int64_t need = (n_max + SEL_SMEM_CAP - 1) / SEL_SMEM_CAP;
    int64_t want = std::max<int64_t>(need, std::min<int64_t>((2LL * ctx->num_sms + rows - 1) / rows,
                                                             n_max / std::max(1, 4 * k)));
    want = std::max<int64_t>(want, 1);
    const int64_t merge_cap = k > 0 ? SEL_SMEM_CAP / k : 1;
    want = std::min<int64_t>(want, merge_cap);
    const size_t per_chunk = (size_t)rows * k * (sizeof(uint32_t) + sizeof(int32_t));
    if (want > 1 && have_ws && ws_bytes / std::max<size_t>(per_chunk, 1) >= (size_t)want &&
        (n_max + want - 1) / want <= SEL_SMEM_CAP) {
        chunks = (int)want;
        chunk_len = (n_max + want - 1) / want;
        smem = true;
        return;
    }
    chunks = 1;
    chunk_len = std::max<int64_t>(n_max, 1);
    smem = n_max <= SEL_SMEM_CAP;
}

// ---------------------------------------------------------------- cluster selection
// Few long rows (the decode pool over 131,072 block maxima, the top-512 over 16,384
// pooled candidates): one thread-block cluster of C CTAs per row.  Each CTA stages its
// contiguous chunk of keys in shared memory.  The three radix digits (12, 10, 10 bits)
// are counted per CTA and summed across the cluster through distributed shared
// memory: each CTA sums one slice of the bins over the cluster, then every CTA reads
// the slice totals and the one slice that holds the threshold, so all find the same
// bin.  Finally each CTA emits its winners in index order, at the offset given by the
// winner and tie counts of the CTAs before it (ties at T go to the lowest indices).
// Every CTA runs the same sequence of cluster barriers whatever the data, so no
// barrier can be left waiting for a CTA that took another path.
constexpr int CL_THREADS = 1024;           // most threads per CTA (chunks of >= 8,192 keys; 512 below)
constexpr int CL_MAX_CHUNK = 16384;        // keys per CTA (64 KB of shared memory)

struct ClShared {
    uint32_t hist[NB_A];                   // this CTA's histogram of the current digit
    uint32_t full[NB_A];                   // the row's histogram (every owner pushes its slice)
    uint32_t wtot[32];
    uint32_t wtot_all;
    uint32_t wgt[32], weq[32];             // per-warp winner / tie counts
    uint32_t gt, eq;                       // this CTA's keys above T / equal to T
    uint32_t total;                        // keys counted by the last search, whole row
    int bin;
    uint32_t above;
    uint32_t off, take, nsel;              // emission: output offset, ties taken, row total
};

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster; release / acquire orders shared memory.
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the word at `p` in the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    return ra;
}
__device__ __forceinline__ uint32_t cl_ld(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
// Sum of the words at offset `off` in the shared memory of CTAs 0..7 (bases b[]): the
// eight loads are issued back to back, one round trip for all.
__device__ __forceinline__ uint32_t cl_sum8(const uint32_t* b, uint32_t off) {
    uint32_t v0, v1, v2, v3, v4, v5, v6, v7;
    asm volatile(
        "ld.shared::cluster.u32 %0, [%8];\n\t"
        "ld.shared::cluster.u32 %1, [%9];\n\t"
        "ld.shared::cluster.u32 %2, [%10];\n\t"
        "ld.shared::cluster.u32 %3, [%11];\n\t"
        "ld.shared::cluster.u32 %4, [%12];\n\t"
        "ld.shared::cluster.u32 %5, [%13];\n\t"
        "ld.shared::cluster.u32 %6, [%14];\n\t"
        "ld.shared::cluster.u32 %7, [%15];"
        : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3), "=r"(v4), "=r"(v5), "=r"(v6), "=r"(v7)
        : "r"(b[0] + off), "r"(b[1] + off), "r"(b[2] + off), "r"(b[3] + off), "r"(b[4] + off), "r"(b[5] + off),
          "r"(b[6] + off), "r"(b[7] + off)
        : "memory");
    return ((v0 + v1) + (v2 + v3)) + ((v4 + v5) + (v6 + v7));
}

__device__ __forceinline__ void cl_st(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ void cl_search_full(ClShared& sh, int nb, uint32_t remaining, int& bin, uint32_t& above);

// Cluster-wide: the bin (of nb, searched from the top) holding the remaining-th
// largest key of the row, and the number of keys in the bins above it, from every
// CTA's local histogram sh.hist.  CTA r sums bins [r*W, r*W+W) over the cluster and
// pushes the sums into every CTA's sh.full, so after one more barrier each CTA holds
// the row's histogram and searches it locally.  sh.total gets the number of keys
// counted; if remaining exceeds it, bin = 0 and above = 0 (the caller takes all).
// base[c] = the cluster address of CTA c's ClShared.  blockDim.x == CL_THREADS.
__device__ void cl_find_bin(ClShared& sh, int nb, uint32_t remaining, uint32_t C, uint32_t rank,
                            const uint32_t* base, int& bin, uint32_t& above) {
    const int W = nb / (int)C;             // bins per slice, <= blockDim
    const uint32_t hist_off = (uint32_t)offsetof(ClShared, hist);
    const uint32_t full_off = (uint32_t)offsetof(ClShared, full);
    cl_sync();                             // every CTA's histogram is complete, and every
                                           // CTA has finished reading its sh.full
    if ((int)threadIdx.x < W) {
        const uint32_t off = 4u * (rank * (uint32_t)W + threadIdx.x);
        uint32_t v = 0u;
        if (C == 8 || C == 16) {
            v = cl_sum8(base, hist_off + off);
            if (C == 16) v += cl_sum8(base + 8, hist_off + off);
        } else {
            for (uint32_t c = 0; c < C; ++c) v += cl_ld(base[c] + hist_off + off);
        }
        for (uint32_t c = 0; c < C; ++c) cl_st(base[c] + full_off + off, v);
    }
    cl_sync();                             // every slice is in every CTA's sh.full
    cl_search_full(sh, nb, remaining, bin, above);
}

// Search sh.full (a whole row's histogram of nb bins) from the top for the bin holding
// the remaining-th largest key: bin, and the keys in the bins above it; sh.total gets
// the keys counted (bin = 0, above = 0 if remaining exceeds it).  nb is a multiple of
// the block size.
__device__ void cl_search_full(ClShared& sh, int nb, uint32_t remaining, int& bin, uint32_t& above) {
    const int per = nb / (int)blockDim.x;
    const int top = nb - 1 - (int)threadIdx.x * per;
    uint32_t loc = 0;
    for (int j = 0; j < per; ++j) loc += sh.full[top - j];
    uint32_t total;
    const uint32_t excl = block_excl_scan_u32(loc, sh, total);
    if (threadIdx.x == 0) {
        sh.bin = 0;
        sh.above = 0u;
        sh.total = total;
    }
    __syncthreads();
    if (excl < remaining && remaining <= excl + loc) {
        uint32_t cum = excl;
        for (int j = 0; j < per; ++j) {
            const uint32_t c = sh.full[top - j];
            if (cum + c >= remaining) {
                sh.bin = top - j;
                sh.above = cum;
                break;
            }
            cum += c;
        }
    }
    __syncthreads();
    bin = sh.bin;
    above = sh.above;
}

// Keys of elements c0 .. c0+n-1 of the row into skey, and the first digit's local
// histogram; values are read four at a time when the chunk is 16-byte aligned.
template <int MODE>
__device__ void cl_stage(const SelArgs& a, int64_t row, int64_t c0, int n, int64_t V, int64_t n_elems,
                         uint32_t* skey, uint32_t* hist) {
    const int tid = threadIdx.x;
    const float* rowp = a.vals + row * a.ld + c0;
    const bool vec = (reinterpret_cast<uintptr_t>(rowp) & 15u) == 0;
    const int nq = vec ? n / 4 : 0;
    for (int base = 0; base < nq; base += (int)blockDim.x * 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = base + j * (int)blockDim.x + tid;
            v[j] = q < nq ? reinterpret_cast<const float4*>(rowp)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = base + j * (int)blockDim.x + tid;
            if (q >= nq) continue;
            const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t kk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                kk[c] = elem_info<MODE>(a, row, c0 + 4 * q + c, V, n_elems).valid ? order_key(f[c]) : 0u;
                if (kk[c]) atomicAdd(&hist[kk[c] >> 20], 1u);
            }
            reinterpret_cast<uint4*>(skey)[q] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
        }
    }
    for (int i = 4 * nq + tid; i < n; i += blockDim.x) {
        const uint32_t key = key_of<MODE>(a, row, c0 + i, V, n_elems);
        skey[i] = key;
        if (key) atomicAdd(&hist[key >> 20], 1u);
    }
}

template <int MODE>
__global__ void __launch_bounds__(CL_THREADS) sel_cluster_kernel(SelArgs a, int chunk) {
    extern __shared__ uint32_t skey[];     // [chunk]
    __shared__ ClShared sh;
    pdl_wait();                            // the scores / block maxima are complete
    const uint32_t C = cl_size(), rank = cl_rank();
    const int64_t row = blockIdx.y;
    const int64_t V = a.nv[row];
    const int64_t n_elems = row_elems<MODE>(a, V);
    const int64_t c0 = (int64_t)rank * chunk;
    const int n = (int)max((int64_t)0, min((int64_t)chunk, n_elems - c0));
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int k = a.k;
    uint32_t base[16];                     // cluster addresses of every CTA's ClShared
#pragma unroll
    for (int c = 0; c < 16; ++c) base[c] = cl_map(&sh, (uint32_t)c < C ? (uint32_t)c : 0u);

    // stage the chunk's keys and count the first digit (bits 31..20)
    for (int i = threadIdx.x; i < NB_A; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    cl_stage<MODE>(a, row, c0, n, V, n_elems, skey, sh.hist);
    __syncthreads();
    int b1, b2, b3;
    uint32_t ab1, ab2, ab3;
    cl_find_bin(sh, NB_A, (uint32_t)k, C, rank, base, b1, ab1);
    const bool take_all = sh.total <= (uint32_t)k;
    uint32_t prefix = (uint32_t)b1 << 20;
    uint32_t rem = take_all ? 0u : (uint32_t)k - ab1;
    // second digit (bits 19..10) over the keys of the threshold bin; the searches run
    // (on empty histograms) even when every key is taken, keeping the barriers uniform
    for (int i = threadIdx.x; i < NB_B; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const uint32_t key = i < n ? skey[i] : 0u;
        hist_add_warp(sh.hist, (key >> 10) & 0x3FFu, !take_all && key != 0u && (key & 0xFFF00000u) == prefix);
    }
    __syncthreads();
    cl_find_bin(sh, NB_B, take_all ? 1u : rem, C, rank, base, b2, ab2);
    prefix |= (uint32_t)b2 << 10;
    rem -= take_all ? 0u : ab2;
    // third digit (bits 9..0)
    for (int i = threadIdx.x; i < NB_B; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const uint32_t key = i < n ? skey[i] : 0u;
        hist_add_warp(sh.hist, key & 0x3FFu, !take_all && key != 0u && (key & 0xFFFFFC00u) == prefix);
    }
    __syncthreads();
    cl_find_bin(sh, NB_B, take_all ? 1u : rem, C, rank, base, b3, ab3);
    prefix |= (uint32_t)b3;
    rem -= take_all ? 0u : ab3;
    // the k-th key T and the number of keys equal to T to take (lowest indices first);
    // take_all: every valid key (keys are never 0)
    const uint32_t T = take_all ? 0u : prefix;
    const uint32_t r_ties = take_all ? 0u : rem;

    // emission, pass 1: per-warp counts over a contiguous segment (32 keys per step)
    const int seg = ((n + nwarps - 1) / nwarps + 31) / 32 * 32;
    const int w0 = wid * seg, w1 = min(n, w0 + seg);
    uint32_t cgt = 0, ceq = 0;
    for (int j = w0; j < w1; j += 32) {
        const int i = j + lane;
        const uint32_t key = i < w1 ? skey[i] : 0u;
        cgt += __popc(__ballot_sync(FULL_MASK, key > T));
        ceq += __popc(__ballot_sync(FULL_MASK, T != 0u && key == T));
    }
    if (lane == 0) {
        sh.wgt[wid] = cgt;
        sh.weq[wid] = ceq;
    }
    __syncthreads();
    if (wid == 0) {
        uint32_t g = lane < nwarps ? sh.wgt[lane] : 0u, e = lane < nwarps ? sh.weq[lane] : 0u;
        uint32_t gi = g, ei = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t ug = __shfl_up_sync(FULL_MASK, gi, o), ue = __shfl_up_sync(FULL_MASK, ei, o);
            if (lane >= o) {
                gi += ug;
                ei += ue;
            }
        }
        if (lane < nwarps) {
            sh.wgt[lane] = gi - g;         // exclusive: before this warp
            sh.weq[lane] = ei - e;
        }
        if (lane == 31) {
            sh.gt = gi;
            sh.eq = ei;
        }
    }
    cl_sync();                              // every CTA's counts are published
    if (wid == 0) {
        // offsets from the CTAs before this one (index order = rank order)
        const uint32_t g = lane < C ? cl_ld(base[lane < C ? lane : 0] + (uint32_t)offsetof(ClShared, gt)) : 0u;
        const uint32_t e = lane < C ? cl_ld(base[lane < C ? lane : 0] + (uint32_t)offsetof(ClShared, eq)) : 0u;
        uint32_t ei = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(FULL_MASK, ei, o);
            if (lane >= o) ei += u;
        }
        const uint32_t ties_before = ei - e;
        const uint32_t take = r_ties > ties_before ? min(r_ties - ties_before, e) : 0u;
        uint32_t sel = g + take, si = sel;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(FULL_MASK, si, o);
            if (lane >= o) si += u;
        }
        if (lane == rank) {
            sh.off = si - sel;
            sh.take = take;
        }
        if (lane == 31) sh.nsel = si;
    }
    __syncthreads();
    // pass 2: write the winners in index order
    {
        const uint32_t off = sh.off, take = sh.take;
        uint32_t gb = sh.wgt[wid], eb = sh.weq[wid];
        const unsigned lt = (1u << lane) - 1u;
        for (int j = w0; j < w1; j += 32) {
            const int i = j + lane;
            const uint32_t key = i < w1 ? skey[i] : 0u;
            const unsigned mg = __ballot_sync(FULL_MASK, key > T);
            const unsigned me = __ballot_sync(FULL_MASK, T != 0u && key == T);
            const uint32_t g_before = gb + __popc(mg & lt), e_before = eb + __popc(me & lt);
            const bool isel = key > T || (T != 0u && key == T && e_before < take);
            if (isel) {
                const int64_t pos = (int64_t)off + g_before + min(e_before, take);
                a.out_idx[row * a.out_len + pos] = (int32_t)elem_info<MODE>(a, row, c0 + i, V, n_elems).id;
                if (a.out_val) a.out_val[row * a.out_len + pos] = a.vals[row * a.ld + c0 + i];
            }
            gb += __popc(mg);
            eb += __popc(me);
        }
    }
    // the rest of the row: the newest visible block (pool), then padding; spread over
    // the cluster's threads
    {
        int64_t filled = sh.nsel;
        if (MODE == SEL_POOL && n_elems > 0) {
            if (rank == 0 && threadIdx.x == 0) a.out_idx[row * a.out_len + filled] = (int32_t)(n_elems - 1);
            ++filled;
        }
        for (int64_t i = filled + (int64_t)rank * blockDim.x + threadIdx.x; i < a.out_len;
             i += (int64_t)C * blockDim.x) {
            a.out_idx[row * a.out_len + i] = -1;
            if (a.out_val) a.out_val[row * a.out_len + i] = -INFINITY;
        }
    }
    pdl_trigger();
    cl_sync();                              // no CTA leaves while another reads its counts
}

// Cluster size for the cluster path, or 0 when it does not apply: few rows, each split
// into chunks of at most CL_MAX_CHUNK keys.  8 CTAs when the chunks fit (measured: the
// cluster barriers of 8 CTAs are cheaper than those of 16), else 16.
int cluster_size_for(csa2_ctx* ctx, int64_t rows, int64_t n_max) {
    if (n_max <= 8192) return 0;           // one CTA stages the row: no cluster barriers
    for (int c : {8, 16}) {
        if (rows * c > ctx->num_sms) return 0;
        if (((n_max + c - 1) / c + 31) / 32 * 32 > CL_MAX_CHUNK) continue;
        return c;
    }
    return 0;
}

template <int MODE>
csa2_status launch_cluster(csa2_ctx* ctx, const SelArgs& a, int64_t rows, int64_t n_max, int C, cudaStream_t s) {
    auto kern = sel_cluster_kernel<MODE>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CL_MAX_CHUNK * 4) !=
                cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return CSA2_ERR_CUDA;
        attr = true;
    }
    const int chunk = (int)(((n_max + C - 1) / C + 31) / 32 * 32);   // 16-byte aligned chunk starts
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)rows, 1);
    cfg.blockDim = dim3(chunk >= 8192 ? 1024 : 512, 1, 1);   // >= the 512 bins of a 12-bit slice at C = 8
    cfg.dynamicSmemBytes = (size_t)chunk * sizeof(uint32_t);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait()
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, a, chunk) != cudaSuccess) return CSA2_ERR_CUDA;
    return csa2_launch_status();
}

// ---------------------------------------------------------------- pool from a histogram
// The decode pool (CSA2 page, «解码器里的分层索引») with the first radix digit already
// counted: the indexer scan adds every visible block maximum's leading 12 key bits to
// a per-row histogram, so the threshold bin of the pool (rank n_keep-1 among the
// blocks other than the newest) and of the top blocks (rank n_top among all blocks)
// are read off that histogram.  One thread-block cluster per row; each CTA loads its
// chunk of block maxima (every load in flight at once, beside the histogram's) and
// classifies them: above the threshold bin -> winner, in it -> candidate.  The
// candidates of the whole row are few (a few hundred on Gaussian scores: a bin is 1/8
// of an octave wide), so every CTA gathers all of them through distributed shared
// memory and ranks its own ones against them in the order (key desc, index asc): a
// candidate wins if fewer than the remaining count rank above it.  Only a threshold
// bin of more than PH_CAP keys takes cluster-wide radix passes (a threshold key T,
// ties at T taken lowest index first).  Each CTA then pushes its winner and tie
// counts into every CTA of the cluster, and after one more cluster barrier emits its
// winners in index order at its offset.  The barrier sequence depends only on the
// row's histogram, so every CTA of a cluster runs the same one.
constexpr int PH_CAP = 2048;               // candidates a selection gathers on every CTA
constexpr int PH_MAX_C = 16;
constexpr int PH_KPT = CL_MAX_CHUNK / CL_THREADS;   // keys a thread loads (16)

struct PoolArgs {
    const float* bmax;        // [rows, ld]
    int64_t ld;
    const int64_t* nv;        // [rows] visible entries
    const uint32_t* hist;     // [rows, NB_A] first-digit counts of the visible block maxima
    int block;
    int n_keep;               // pool size: the newest block + n_keep - 1 others
    int32_t* out_pool;        // [rows, n_keep]
    int n_top;                // 0: no top list (with ENTRY: k, the blocks that hold the top-k)
    int32_t* out_top;         // [rows, n_top] or NULL
    unsigned int* st;
    // ENTRY: the row's top-k entries from the stored scores of its k best blocks
    const float* scores;      // [rows, n_ent]
    int64_t n_ent;            // row stride of scores (>= ld * block)
    int k;
    int32_t* out_idx;         // [rows, k]
    float* out_val;           // [rows, k] or NULL
};

struct PhShared {
    uint32_t nloc[2];                      // candidates in this CTA's list, per selection
    uint32_t start[PH_MAX_C + 1];          // the gathered list: where each CTA's candidates begin
    uint32_t cnt[2][PH_MAX_C][2];          // pushed by every CTA: its (winners, ties at T), per selection
    uint32_t rem[2];                       // ties at T to take (cluster-wide radix passes only)
    uint32_t tkey;                         // ENTRY: the smallest block maximum among the best blocks
    uint32_t ecnt;                         // ENTRY: entry candidates pushed into this CTA
    uint32_t ewin[PH_MAX_C];               // ENTRY: every CTA's number of winning entries
    uint32_t nown;                         // ENTRY: this CTA's best blocks
    uint32_t tmin_local;                   // ENTRY: the smallest maximum among this CTA's in-bin best blocks
    uint32_t tmin[PH_MAX_C];               // ENTRY: every CTA's tmin_local (pushed)
    uint32_t ndense;                       // ENTRY: received entries scoring at least the threshold
    uint32_t nwin;                         // ENTRY: this CTA's winning entries
    uint32_t nown_e;                       // ENTRY: received entries of this CTA's chunk
    uint32_t wsum[2][32];                  // threshold search: per-warp bin sums (pool, best blocks)
    int sbin[2];                           // threshold search: the bin, the keys above it, the keys in it
    uint32_t sabove[2], sm[2];
};
constexpr int PH_ECAP = 8192;              // ENTRY: entry candidates a CTA can receive (64 KB)
constexpr int PH_WCAP = 1024;              // ENTRY: winners emitted from a list (more: from the bitmap)
// ENTRY reuses the two candidate-list arrays once the block selections are done:
// `all` (sized for max(2 * PH_CAP, k * block) entries) holds the received entries at or
// above the threshold (at most k * block of them: the entries of the k best blocks),
// `loc` the bitmap of a chunk's entries; the receive buffer holds PH_ECAP entries, so
// k * block <= PH_ECAP.
static_assert(2 * PH_CAP <= PH_ECAP, "every entry of the best blocks fits the receive buffer");
// capacity of `all` for k best blocks of `block` entries
__host__ __device__ inline int ph_dense_cap(int k, int block) { return k * block > 2 * PH_CAP ? k * block : 2 * PH_CAP; }

// Ordered emission of one selection from the CTA's bitmaps: winners (bmW) in index
// order, ties (bmE) while fewer than `quota` have been taken, at out[off + rank].
__device__ __noinline__ void ph_emit(const uint32_t* bmW, const uint32_t* bmE, int nwords, int64_t c0, uint32_t off,
                        uint32_t quota, int32_t* out, uint32_t out_len, ClShared& sh) {
    const int tid = threadIdx.x;
    const int per = (nwords + (int)blockDim.x - 1) / (int)blockDim.x;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    uint32_t cg = 0, ce = 0;
    for (int w = w0; w < w1; ++w) {
        cg += __popc(bmW[w]);
        ce += __popc(bmE[w]);
    }
    uint32_t tot;
    uint32_t gb = block_excl_scan_u32(cg, sh, tot);
    uint32_t eb = block_excl_scan_u32(ce, sh, tot);
    for (int w = w0; w < w1; ++w) {
        const uint32_t wg = bmW[w], we = bmE[w];
        uint32_t bits = wg | we;
        while (bits) {
            const int j = __ffs(bits) - 1;
            bits &= bits - 1;
            const int32_t id = (int32_t)(c0 + w * 32 + j);
            if ((wg >> j) & 1u) {
                const uint32_t pos = off + gb + min(eb, quota);
                if (pos < out_len) out[pos] = id;
                ++gb;
            } else {
                if (eb < quota && off + gb + eb < out_len) out[off + gb + eb] = id;
                ++eb;
            }
        }
    }
}

// Remote atomic add in CTA `rank`'s shared memory (cluster address from cl_map).
__device__ __forceinline__ uint32_t cl_atomic_add(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

// One selection pass over bitmap words in index order: thread t owns a run of words;
// bit j of word w (id base + 32 w + j) goes to out[off + its rank] while below out_len.
__device__ __noinline__ void ph_emit_bits(const uint32_t* bm, int nwords, int64_t base, uint32_t off, int32_t* out,
                             float* outv, const float* vals, uint32_t out_len, ClShared& sh) {
    const int tid = threadIdx.x;
    const int per = (nwords + (int)blockDim.x - 1) / (int)blockDim.x;
    const int w0 = tid * per, w1 = min(nwords, w0 + per);
    uint32_t cg = 0;
    for (int w = w0; w < w1; ++w) cg += __popc(bm[w]);
    uint32_t tot;
    uint32_t pos = off + block_excl_scan_u32(cg, sh, tot);
    for (int w = w0; w < w1; ++w) {
        uint32_t bits = bm[w];
        while (bits) {
            const int j = __ffs(bits) - 1;
            bits &= bits - 1;
            if (pos < out_len) {
                const int64_t id = base + w * 32 + j;
                out[pos] = (int32_t)id;
                if (outv) outv[pos] = vals[id];
            }
            ++pos;
        }
    }
}

// The threshold bins of both selections, searched from the top of the row's histogram
// (NB_A bins in `full`): index 0 the pool (rank kP among the blocks other than the
// newest, whose bin knew_bin counts one block less), index 1 the best blocks (rank kT);
// a rank of 0 skips that search.  Thread t holds bins NB_A-1-4t .. NB_A-4-4t; the warps'
// sums meet in shared memory and the thread whose bins hold the rank walks them.  Each
// result: the bin, the keys in the bins above it, the keys in it (bin 0, 0, 0 when the
// rank exceeds the count).  Two block barriers; blockDim.x * 4 == NB_A.
__device__ __noinline__ void ph_search2(const uint32_t* full, uint32_t knew_bin, uint32_t kP, uint32_t kT,
                                        PhShared& px) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int top = NB_A - 1 - 4 * tid;
    const uint4 q = *reinterpret_cast<const uint4*>(full + top - 3);
    const uint32_t cT[4] = {q.w, q.z, q.y, q.x};        // bins top, top-1, top-2, top-3
    uint32_t cP[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cP[j] = cT[j] - ((uint32_t)(top - j) == knew_bin ? 1u : 0u);
    const uint32_t sT = (cT[0] + cT[1]) + (cT[2] + cT[3]), sP = (cP[0] + cP[1]) + (cP[2] + cP[3]);
    uint32_t iT = sT, iP = sP;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t uT = __shfl_up_sync(FULL_MASK, iT, o), uP = __shfl_up_sync(FULL_MASK, iP, o);
        if (lane >= o) {
            iT += uT;
            iP += uP;
        }
    }
    if (lane == 31) {
        px.wsum[0][wid] = iP;
        px.wsum[1][wid] = iT;
    }
    if (tid < 2) {
        px.sbin[tid] = 0;
        px.sabove[tid] = 0u;
        px.sm[tid] = 0u;
    }
    __syncthreads();
    // keys in the warps' bins above this warp's (every warp scans the 32 sums)
    uint32_t wP = px.wsum[0][lane], wT = px.wsum[1][lane];
    uint32_t jP = wP, jT = wT;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t uT = __shfl_up_sync(FULL_MASK, jT, o), uP = __shfl_up_sync(FULL_MASK, jP, o);
        if (lane >= o) {
            jT += uT;
            jP += uP;
        }
    }
    const uint32_t preP = __shfl_sync(FULL_MASK, jP - wP, wid), preT = __shfl_sync(FULL_MASK, jT - wT, wid);
    const uint32_t exP = preP + iP - sP, exT = preT + iT - sT;
    if (kT > 0u && exT < kT && kT <= exT + sT) {
        uint32_t cum = exT;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (cum + cT[j] >= kT) {
                px.sbin[1] = top - j;
                px.sabove[1] = cum;
                px.sm[1] = cT[j];
                break;
            }
            cum += cT[j];
        }
    }
    if (kP > 0u && exP < kP && kP <= exP + sP) {
        uint32_t cum = exP;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (cum + cP[j] >= kP) {
                px.sbin[0] = top - j;
                px.sabove[0] = cum;
                px.sm[0] = cP[j];
                break;
            }
            cum += cP[j];
        }
    }
    __syncthreads();
}

// Bucket of an entry (flipped (key, index) value): min(1023, (key >> shift) - base),
// 0 below base -- non-decreasing in the key, so any bucket above the one holding the
// r-th largest entry holds only entries ranked above it.
__device__ __forceinline__ int ph_bucket(uint64_t x, int shift, uint32_t base) {
    const uint32_t k = (uint32_t)(x >> 32) >> shift;
    return k <= base ? 0 : (int)min(k - base, 1023u);
}

// The bucket (of 1,024) holding the r-th largest of the mm entries of A (flipped
// values), searched from the top; -1 if r exceeds mm.  blockDim.x == 1024.
__device__ __noinline__ int ph_bucket_of_rank(const uint64_t* A, uint32_t mm, uint32_t r, int shift, uint32_t base,
                                              ClShared& sh, PhShared& px) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t* h = sh.hist;
    h[tid] = 0u;
    if (tid == 0) px.sbin[0] = -1;
    __syncthreads();
    for (uint32_t j = tid; j < mm; j += CL_THREADS) atomicAdd(&h[ph_bucket(A[j], shift, base)], 1u);
    __syncthreads();
    // thread t holds bucket 1023 - t: the entries above it are the sum over the threads before it
    const int b = CL_THREADS - 1 - tid;
    const uint32_t c = h[b];
    uint32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(FULL_MASK, inc, o);
        if (lane >= o) inc += u;
    }
    if (lane == 31) px.wsum[0][wid] = inc;
    __syncthreads();
    const uint32_t ws = px.wsum[0][lane];
    uint32_t wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(FULL_MASK, wi, o);
        if (lane >= o) wi += u;
    }
    const uint32_t ex = __shfl_sync(FULL_MASK, wi - ws, wid) + inc - c;
    if (ex < r && r <= ex + c) px.sbin[0] = b;
    __syncthreads();
    return px.sbin[0];
}

// The winners among this CTA's candidates of a threshold bin.  A: every CTA's
// candidates of the bin (mm of them, flipped so that larger is earlier in the order
// key desc, index asc); own: this CTA's nl candidates (unflipped); r: the winners
// still to take from the bin.  Bucketed by the next 10 key bits: own candidates above
// the bucket of the r-th win, below it lose, and those in it are ranked against all
// of A.  Winners set their bit in W (chunk offset from c0); with track_min,
// px.tmin_local gets the smallest winning key.  blockDim.x == 1024.
__device__ __noinline__ void ph_rank_bin(const uint64_t* A, uint32_t mm, const uint64_t* own, uint32_t nl, uint32_t r,
                                         int64_t c0, uint32_t* W, bool track_min, ClShared& sh, PhShared& px) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t base = ((uint32_t)(A[0] >> 32) >> 20) << 10;   // the bin's keys share their top 12 bits
    const int sb = mm ? ph_bucket_of_rank(A, mm, r, 10, base, sh, px) : -1;
    auto win = [&](uint64_t x) {
        const uint32_t li = (uint32_t)((int64_t)(uint32_t)(x ^ 0xFFFFFFFFull) - c0);
        atomicOr(&W[li >> 5], 1u << (li & 31));
        if (track_min) atomicMin(&px.tmin_local, (uint32_t)(x >> 32));
    };
    for (uint32_t ci = tid; ci < nl; ci += CL_THREADS) {
        const uint64_t x = own[ci] ^ 0xFFFFFFFFull;
        if (ph_bucket(x, 10, base) > sb) win(x);
    }
    // the bucket of the r-th: a warp per own candidate in it, ranked against all of A
    for (uint32_t ci = wid; ci < nl; ci += CL_THREADS / 32) {
        const uint64_t x = own[ci] ^ 0xFFFFFFFFull;
        if (ph_bucket(x, 10, base) != sb) continue;              // the same for the whole warp
        uint32_t ahead = 0u;
#pragma unroll 4
        for (uint32_t j = lane; j < mm; j += 32) ahead += A[j] > x;
        ahead = __reduce_add_sync(FULL_MASK, ahead);
        if (lane == 0 && ahead < r) win(x);
    }
}

template <bool ENTRY>
__global__ void __launch_bounds__(CL_THREADS) pool_hist_kernel(PoolArgs a, int chunk) {
    extern __shared__ __align__(16) uint32_t dyn[];
    __shared__ __align__(16) ClShared sh;
    __shared__ PhShared px;
    pdl_wait();                            // the block maxima, histogram and scores are complete
    const uint32_t C = cl_size(), rank = cl_rank();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t row = blockIdx.y;
    const int64_t V = a.nv[row];
    int64_t nb = V > 0 ? (V + a.block - 1) / a.block : 0;
    if (nb > a.ld) {
        if (tid == 0 && rank == 0) csa2_flag(a.st, CSA2_DEVBIT_RANGE);
        nb = a.ld;
    }
    const bool doT = ENTRY || (a.out_top != nullptr && a.n_top > 0);
    const bool allP = nb <= a.n_keep, allT = !doT || nb <= a.n_top;
    int32_t* outP = a.out_pool + row * a.n_keep;
    int32_t* outT = a.out_top ? a.out_top + row * a.n_top : nullptr;
    const int bd = CL_THREADS;
    // every visible block fits: ascending ids, then -1
    if (allP)
        for (int64_t i = (int64_t)rank * bd + tid; i < a.n_keep; i += (int64_t)C * bd) outP[i] = i < nb ? (int32_t)i : -1;
    if (outT && allT)
        for (int64_t i = (int64_t)rank * bd + tid; i < a.n_top; i += (int64_t)C * bd) outT[i] = i < nb ? (int32_t)i : -1;
    if (!ENTRY && allP && allT) {          // the same for every CTA of the row: no barrier used
        pdl_trigger();
        return;
    }
    // every load of the phase in flight together: this thread's keys (key i of the
    // chunk is loaded by thread i % 1024), the histogram, the newest block's maximum
    const int64_t newest = nb - 1;
    const int64_t c0 = (int64_t)rank * chunk;
    const int n = (int)max((int64_t)0, min((int64_t)chunk, nb - c0));
    const float* rowp = a.bmax + row * a.ld + c0;
    float v[PH_KPT];
#pragma unroll
    for (int j = 0; j < PH_KPT; ++j) {
        const int i = tid + j * bd;
        v[j] = i < n ? rowp[i] : 0.0f;
    }
    const bool need_hist = !allP || !allT;
    const uint32_t* hrow = a.hist + row * NB_A;
    uint32_t hv[NB_A / CL_THREADS];
#pragma unroll
    for (int j = 0; j < NB_A / CL_THREADS; ++j) hv[j] = need_hist ? hrow[tid + j * bd] : 0u;
    const uint32_t knew = nb > 0 ? order_key(a.bmax[row * a.ld + newest]) : 0u;
#pragma unroll
    for (int j = 0; j < NB_A / CL_THREADS; ++j) sh.full[tid + j * bd] = hv[j];
    if (tid < 2) px.nloc[tid] = 0u;
    if (tid == 0) {
        px.ecnt = 0u;
        px.tkey = 1u;                      // take-all: every valid key (keys are never 0)
        px.tmin_local = 0xFFFFFFFFu;
    }
    __syncthreads();
    // the threshold bins of both selections
    const uint32_t k[2] = {(uint32_t)a.n_keep - 1u, (uint32_t)a.n_top};
    const bool act[2] = {!allP, !allT};
    // (the newest block is not among the pool's candidates: its bin counts one less)
    ph_search2(sh.full, knew >> 20, act[0] ? k[0] : 0u, act[1] ? k[1] : 0u, px);
    int bin[2] = {px.sbin[0], px.sbin[1]};
    uint32_t above[2] = {px.sabove[0], px.sabove[1]}, m[2] = {px.sm[0], px.sm[1]};
    // classify: the 32 keys of word w = i / 32 are lanes of one warp in one step
    const int cw = chunk / 32;
    const int nwords = (n + 31) / 32;
    const int skey_words = ENTRY ? max(chunk, 2 * PH_ECAP) : chunk;
    uint32_t* skey = dyn;                                  // [skey_words]; ENTRY: then the received entries
    uint32_t* bmW = dyn + skey_words;                      // [2][cw]
    uint32_t* bmE = bmW + 2 * cw;                          // [2][cw]
    uint64_t* loc = reinterpret_cast<uint64_t*>(bmE + 2 * cw);   // [2][PH_CAP] this CTA's candidates
    uint64_t* all = loc + 2 * PH_CAP;                      // [2][PH_CAP] every CTA's, gathered (ENTRY: more)
    const uint32_t dcap = ENTRY ? (uint32_t)ph_dense_cap(a.k, a.block) : 2u * PH_CAP;
    const unsigned lt = (1u << lane) - 1u;
    // the chunk's keys into shared memory (key i from thread i % 1024: coalesced loads)
#pragma unroll
    for (int j = 0; j < PH_KPT; ++j) {
        const int i = tid + j * bd;
        if (i >= chunk) break;
        skey[i] = i < n ? order_key(v[j]) : 0u;
    }
    __syncthreads();
    // classify: two threads per word of 32 keys (threads 2w and 2w+1 take its halves),
    // each half read as four 16-byte pieces starting at a word-dependent piece (the
    // lanes of a warp then spread over the banks); the halves' bits meet by shuffle
    const int np2 = 2 * nwords;
    for (int p0 = 0; p0 < np2; p0 += bd) {                 // the same bounds for every thread
        const int pw = p0 + tid;
        const bool on = pw < np2;
        const int w = pw >> 1, h = pw & 1;
        uint32_t g0 = 0u, g1 = 0u;
        if (on) {
            uint32_t e0 = 0u, e1 = 0u, vm = 0u;
            // not unrolled: each CTA runs this once, from a cold instruction cache, and
            // straight-line code there costs more in instruction fetch than the loop does
#pragma unroll 1
            for (int t = 0; t < 4; ++t) {
                const int q = 4 * h + ((t + w) & 3);
                const uint4 k4 = *reinterpret_cast<const uint4*>(skey + w * 32 + 4 * q);
                const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t key = kk[c], bit = 1u << (4 * q + c);
                    const int d = (int)(key >> 20);
                    if (key != 0u) {
                        vm |= bit;
                        if (d > bin[0]) g0 |= bit;
                        if (d == bin[0]) e0 |= bit;
                        if (d > bin[1]) g1 |= bit;
                        if (d == bin[1]) e1 |= bit;
                    }
                }
            }
            const int64_t nw_ = newest - c0 - (int64_t)w * 32;      // the newest block is not a pool candidate
            const uint32_t notnew = (nw_ >= 0 && nw_ < 32) ? ~(1u << nw_) : 0xFFFFFFFFu;
            g0 = act[0] ? g0 & notnew : 0u;
            e0 = act[0] ? e0 & notnew : 0u;
            // ENTRY with every block among the best: every visible block of the chunk is one
            g1 = act[1] ? g1 : (ENTRY ? vm : 0u);
            e1 = act[1] ? e1 : 0u;
            // the threshold bins' keys go to this CTA's candidate lists (key, index)
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                uint32_t e = s2 == 0 ? e0 : e1;
                if (!e) continue;
                uint32_t o = atomicAdd(&px.nloc[s2], (uint32_t)__popc(e));
                while (e) {
                    const int j = __ffs(e) - 1;
                    e &= e - 1;
                    if (o < PH_CAP) loc[s2 * PH_CAP + o] = ((uint64_t)skey[w * 32 + j] << 32) | (uint32_t)(c0 + w * 32 + j);
                    ++o;
                }
            }
        }
        g0 |= __shfl_xor_sync(FULL_MASK, g0, 1);
        g1 |= __shfl_xor_sync(FULL_MASK, g1, 1);
        if (on && h == 0) {
            bmW[w] = g0;
            bmW[cw + w] = g1;
            bmE[w] = 0u;
            bmE[cw + w] = 0u;
        }
    }
    cl_sync();                             // (1) every CTA's candidate list is complete
    bool any_radix = false;
#pragma unroll 1
    for (int s2 = 0; s2 < 2; ++s2) {
        if (!act[s2]) continue;
        uint32_t* W = bmW + s2 * cw;
        uint32_t* E = bmE + s2 * cw;
        const uint32_t r = k[s2] - above[s2];              // winners still to find in the bin
        uint32_t rem_ties = 0u;
        if (m[s2] <= (uint32_t)PH_CAP) {
            // gather every CTA's candidates (one remote load each, all in flight), then
            // rank this CTA's own candidates against them: (key desc, index asc)
            uint64_t* A = all + s2 * PH_CAP;
            if (tid < 32) {
                const uint32_t nc = tid < (int)C ? min(cl_ld(cl_map(&px, tid) + (uint32_t)offsetof(PhShared, nloc) +
                                                             4u * s2), (uint32_t)PH_CAP) : 0u;
                uint32_t incl = nc;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t u = __shfl_up_sync(FULL_MASK, incl, o);
                    if (tid >= o) incl += u;
                }
                if (tid <= (int)C) px.start[tid] = incl - nc;     // start[C]: the total
            }
            __syncthreads();
            const uint32_t mm = min(px.start[C], (uint32_t)PH_CAP);
            for (uint32_t j = tid; j < mm; j += bd) {
                uint32_t c = 0;
                while (c + 1 < C && j >= px.start[c + 1]) ++c;
                const uint32_t src = cl_map(loc + s2 * PH_CAP, c) + 8u * (j - px.start[c]);
                uint32_t lo, hi;
                asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(src) : "memory");
                A[j] = (((uint64_t)hi << 32) | lo) ^ 0xFFFFFFFFull;   // larger = earlier in the order
            }
            __syncthreads();
            // ENTRY: the smallest best-block maximum is the smallest in-bin winner of the
            // whole row, the minimum over the CTAs of each one's local minimum
            ph_rank_bin(A, mm, loc + s2 * PH_CAP, min(px.nloc[s2], (uint32_t)PH_CAP), r, c0, W,
                        ENTRY && s2 == 1, sh, px);
        } else {
            // a crowded threshold bin: the remaining two digits cluster-wide, then the
            // ties at T by index
            any_radix = true;
            uint32_t prefix = (uint32_t)bin[s2] << 20, rr = r;
            for (int pass = 0; pass < 2; ++pass) {
                const int shift = pass == 0 ? 10 : 0;
                const uint32_t pm = pass == 0 ? 0xFFF00000u : 0xFFFFFC00u;
                for (int i = tid; i < NB_B; i += bd) sh.hist[i] = 0u;
                __syncthreads();
                for (int i0 = 0; i0 < nwords * 32; i0 += bd) {
                    const int i = i0 + tid;
                    const uint32_t key = i < nwords * 32 ? skey[i] : 0u;
                    const bool ok = key != 0u && (key & pm) == prefix && !(s2 == 0 && c0 + i == newest);
                    hist_add_warp(sh.hist, (key >> shift) & 0x3FFu, ok);
                }
                __syncthreads();
                uint32_t base[PH_MAX_C];
#pragma unroll
                for (int c = 0; c < PH_MAX_C; ++c) base[c] = cl_map(&sh, (uint32_t)c < C ? (uint32_t)c : 0u);
                int b2;
                uint32_t ab;
                cl_find_bin(sh, NB_B, rr, C, rank, base, b2, ab);
                prefix |= (uint32_t)b2 << shift;
                rr -= ab;
            }
            rem_ties = rr;
            for (int i = tid; i < n; i += bd) {
                const uint32_t key = skey[i];
                if (key == 0u || (key >> 20) != (uint32_t)bin[s2] || (s2 == 0 && c0 + i == newest)) continue;
                if (key > prefix) atomicOr(&W[i >> 5], 1u << (i & 31));
                else if (key == prefix) atomicOr(&E[i >> 5], 1u << (i & 31));
            }
            if (ENTRY && s2 == 1 && tid == 0) px.tkey = prefix;
        }
        if (s2 == 0 && newest >= c0 && newest < c0 + n) {   // the pool always keeps the newest block
            const int li = (int)(newest - c0);
            if (tid == 0) atomicOr(&W[li >> 5], 1u << (li & 31));
        }
        __syncthreads();
        // this CTA's winner and tie counts, pushed into every CTA of the cluster
        uint32_t cwin = 0u, ctie = 0u;
        for (int w = tid; w < nwords; w += bd) {
            cwin += __popc(W[w]);
            ctie += __popc(E[w]);
        }
        cwin = __reduce_add_sync(FULL_MASK, cwin);
        ctie = __reduce_add_sync(FULL_MASK, ctie);
        __shared__ uint32_t wsum[2][CL_THREADS / 32];
        if (lane == 0) {
            wsum[0][wid] = cwin;
            wsum[1][wid] = ctie;
        }
        if (tid == 0) px.rem[s2] = rem_ties;
        __syncthreads();
        if (tid < (int)C) {
            uint32_t tw = 0u, tt = 0u;
            for (int i = 0; i < CL_THREADS / 32; ++i) {
                tw += wsum[0][i];
                tt += wsum[1][i];
            }
            const uint32_t dst = cl_map(&px.cnt[s2][rank][0], (uint32_t)tid);
            cl_st(dst, tw);
            cl_st(dst + 4u, tt);
            if (ENTRY && s2 == 1) cl_st(cl_map(&px.tmin[rank], (uint32_t)tid), px.tmin_local);
        }
        __syncthreads();
    }
    if (ENTRY) {
        // ---- the row's top-k entries: every entry of the best blocks that scores at
        // least the smallest best-block maximum is a candidate.  Each CTA pushes the
        // visible entries of its best blocks at or above the best blocks' threshold bin
        // into every CTA (the exact threshold is known only after the next barrier),
        // then each filters the received ones and ranks its own candidates against the
        // rest
        uint32_t* W = bmW + cw;
        if (any_radix) {
            // the crowded case: the ties at T taken (lowest index first) become best
            // blocks once every CTA's counts are in; the barrier also ends every use of
            // skey before entries are pushed into it
            cl_sync();
            if (act[1] && m[1] > (uint32_t)PH_CAP && tid == 0) {
                uint32_t tb = 0u;
                for (uint32_t c = 0; c < rank; ++c) tb += px.cnt[1][c][1];
                const uint32_t rem = px.rem[1];
                uint32_t quota = rem > tb ? min(rem - tb, px.cnt[1][rank][1]) : 0u;
                const uint32_t* E = bmE + cw;
                for (int w = 0; w < nwords && quota; ++w) {
                    uint32_t e = E[w];
                    while (e && quota) {
                        const int j = __ffs(e) - 1;
                        e &= e - 1;
                        W[w] |= 1u << j;
                        --quota;
                    }
                }
            }
            __syncthreads();
        }
        // this CTA's best blocks, compacted into `all` (free now) in index order
        uint32_t* blist = reinterpret_cast<uint32_t*>(all);
        {
            const int per = (nwords + bd - 1) / bd;
            const int w0 = tid * per, w1 = min(nwords, w0 + per);
            uint32_t cnt = 0;
            for (int w = w0; w < w1; ++w) cnt += __popc(W[w]);
            uint32_t tot;
            uint32_t o = block_excl_scan_u32(cnt, sh, tot);
            for (int w = w0; w < w1; ++w) {
                uint32_t bits = W[w];
                while (bits) {
                    const int j = __ffs(bits) - 1;
                    bits &= bits - 1;
                    if (o < 2u * PH_CAP) blist[o] = (uint32_t)(w * 32 + j);
                    ++o;
                }
            }
            if (tid == 0) px.nown = min(tot, 2u * (uint32_t)PH_CAP);
        }
        __syncthreads();
        const uint32_t nown = px.nown;
        const float* srow = a.scores + row * a.n_ent;
        // the threshold is the maximum of a best block, so at least the best blocks'
        // threshold bin's lower edge: an entry below that edge is never a candidate
        const uint32_t edge = (uint32_t)bin[1] << 20;
        for (uint32_t t0 = 0; t0 < nown * (uint32_t)a.block; t0 += bd) {
            const uint32_t t = t0 + tid;
            bool keep = false;
            uint32_t key = 0u;
            int64_t e = 0;
            if (t < nown * (uint32_t)a.block) {
                e = (c0 + blist[t / a.block]) * a.block + t % a.block;
                if (e < V) {
                    key = order_key(srow[e]);
                    keep = key >= edge;
                }
            }
            const unsigned km = __ballot_sync(FULL_MASK, keep);
            if (!km) continue;
            const uint64_t cand = ((uint64_t)key << 32) | (uint32_t)e;
            // one slot reservation per destination CTA, lanes 0 .. C-1 at once
            uint32_t rsv = 0u;
            if (lane < (int)C) rsv = cl_atomic_add(cl_map(&px.ecnt, (uint32_t)lane), (uint32_t)__popc(km));
            for (uint32_t c = 0; c < C; ++c) {
                const uint32_t o = __shfl_sync(FULL_MASK, rsv, (int)c) + __popc(km & lt);
                if (keep && o < (uint32_t)PH_ECAP) {
                    const uint32_t dst = cl_map(skey, c) + 8u * o;
                    asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(dst), "r"((uint32_t)cand),
                                 "r"((uint32_t)(cand >> 32)) : "memory");
                }
            }
        }
    }
    cl_sync();                             // (2) every CTA's counts (and entry candidates) are in every CTA
#pragma unroll 1
    for (int s2 = 0; s2 < 2; ++s2) {
        if (!act[s2]) continue;
        if (s2 == 1 && !outT) continue;
        uint32_t off = 0u, ties_before = 0u, total = 0u, quota = 0u;
        const uint32_t rem = px.rem[s2];
        for (uint32_t c = 0; c < C; ++c) {
            const uint32_t wc = px.cnt[s2][c][0], tc = px.cnt[s2][c][1];
            const uint32_t take = rem > ties_before ? min(rem - ties_before, tc) : 0u;
            if (c < rank) off += wc + take;
            if (c == rank) quota = take;
            total += wc + take;
            ties_before += tc;
        }
        int32_t* out = s2 == 0 ? outP : outT;
        const int out_len = s2 == 0 ? a.n_keep : a.n_top;
        ph_emit(bmW + s2 * cw, bmE + s2 * cw, nwords, c0, off, quota, out, (uint32_t)out_len, sh);
        for (int64_t i = (int64_t)total + (int64_t)rank * bd + tid; i < out_len; i += (int64_t)C * bd) out[i] = -1;
        __syncthreads();
    }
    if (ENTRY) {
        // rank this CTA's own entry candidates (entries of its chunk) against all
        // received ones; the winners go to a bitmap over the chunk's entries (in `loc`,
        // which no CTA reads after barrier (2))
        __shared__ uint32_t wlist[PH_WCAP];  // this CTA's winners (entry offsets in the chunk), unordered
        __shared__ uint32_t olist[PH_WCAP];  // where this CTA's own entries sit in `dense`
        const uint32_t me = min(px.ecnt, (uint32_t)PH_ECAP);
        const uint64_t* ec = reinterpret_cast<const uint64_t*>(skey);
        uint32_t* ebm = reinterpret_cast<uint32_t*>(loc);
        const int ew = (chunk * a.block + 31) / 32;
        for (int i = tid; i < ew; i += bd) ebm[i] = 0u;
        // the threshold: the minimum of the CTAs' smallest in-bin winners (a crowded bin:
        // T itself; every block among the best: any valid key)
        uint32_t tkey = px.tkey;
        if (act[1] && m[1] <= (uint32_t)PH_CAP) {
            tkey = 0xFFFFFFFFu;
            for (uint32_t c = 0; c < C; ++c) tkey = min(tkey, px.tmin[c]);
        }
        if (tid == 0) {
            px.ndense = 0u;
            px.nwin = 0u;
            px.nown_e = 0u;
        }
        __syncthreads();
        const int64_t e0 = c0 * a.block, e1 = (c0 + n) * a.block;
        // the received entries at or above the threshold, as (order value, entry), in `all`
        uint64_t* dense = all;
        for (uint32_t j0 = 0; j0 < me; j0 += bd) {
            const uint32_t j = j0 + tid;
            const bool keep = j < me && (uint32_t)(ec[j] >> 32) >= tkey;
            const unsigned km = __ballot_sync(FULL_MASK, keep);
            if (!km) continue;
            uint32_t o = 0u;
            if (lane == 0) o = atomicAdd(&px.ndense, (uint32_t)__popc(km));
            o = __shfl_sync(FULL_MASK, o, 0) + __popc(km & lt);
            if (keep && o < dcap) {
                dense[o] = ec[j] ^ 0xFFFFFFFFull;     // larger = earlier in the order
                const int64_t e = (int64_t)(uint32_t)ec[j];
                if (e >= e0 && e < e1) {
                    const uint32_t q = atomicAdd(&px.nown_e, 1u);
                    if (q < (uint32_t)PH_WCAP) olist[q] = o;
                }
            }
        }
        __syncthreads();
        const uint32_t md = min(px.ndense, dcap);
        // the winners rank below k among the received entries: bucketed by key bits 29..15
        // above the threshold bin's edge (every received key is at least that edge), own
        // entries above the bucket of the k-th win, and those in it are ranked against all
        // (from the list of own entries, else picked out of all received ones)
        const uint32_t ebase = (uint32_t)bin[1] << 5;
        const int sbe = ph_bucket_of_rank(dense, md, (uint32_t)a.k, 15, ebase, sh, px);
        const uint32_t no = px.nown_e;
        const bool listed = no <= (uint32_t)PH_WCAP;
        auto ewin = [&](int64_t e) {
            const uint32_t li = (uint32_t)(e - e0);
            atomicOr(&ebm[li >> 5], 1u << (li & 31));
            const uint32_t o = atomicAdd(&px.nwin, 1u);
            if (o < (uint32_t)PH_WCAP) wlist[o] = li;
        };
        for (uint32_t ci = tid; ci < (listed ? no : md); ci += CL_THREADS) {
            const uint64_t x = dense[listed ? olist[ci] : ci];
            const int64_t e = (int64_t)(uint32_t)(x ^ 0xFFFFFFFFull);
            if (e >= e0 && e < e1 && ph_bucket(x, 15, ebase) > sbe) ewin(e);
        }
        for (uint32_t ci = wid; ci < (listed ? no : md); ci += CL_THREADS / 32) {
            const uint64_t x = dense[listed ? olist[ci] : ci];
            const int64_t e = (int64_t)(uint32_t)(x ^ 0xFFFFFFFFull);
            if (e < e0 || e >= e1 || ph_bucket(x, 15, ebase) != sbe) continue;   // the same for the whole warp
            uint32_t ahead = 0u;
#pragma unroll 4
            for (uint32_t j = lane; j < md; j += 32) ahead += dense[j] > x;
            ahead = __reduce_add_sync(FULL_MASK, ahead);
            if (lane == 0 && ahead < (uint32_t)a.k) ewin(e);
        }
        __syncthreads();
        const uint32_t nwin = px.nwin;
        if (tid < (int)C) cl_st(cl_map(&px.ewin[rank], (uint32_t)tid), nwin);
        cl_sync();                         // (3) every CTA's winner count is in every CTA
        uint32_t off = 0u, total = 0u;
        for (uint32_t c = 0; c < C; ++c) {
            if (c < rank) off += px.ewin[c];
            total += px.ewin[c];
        }
        int32_t* oi = a.out_idx + row * a.k;
        float* ov = a.out_val ? a.out_val + row * a.k : nullptr;
        if (nwin <= (uint32_t)PH_WCAP) {
            // few winners: each one's place among this CTA's is the count of smaller ids
            const float* vals = a.scores + row * a.n_ent;
            for (uint32_t i = tid; i < nwin; i += bd) {
                const uint32_t li = wlist[i];
                uint32_t pos = 0u;
                for (uint32_t j = 0; j < nwin; ++j) pos += wlist[j] < li;
                pos += off;
                if (pos < (uint32_t)a.k) {
                    const int64_t id = e0 + li;
                    oi[pos] = (int32_t)id;
                    if (ov) ov[pos] = vals[id];
                }
            }
        } else {
            ph_emit_bits(ebm, ew, e0, off, oi, ov, a.scores + row * a.n_ent, (uint32_t)a.k, sh);
        }
        for (int64_t i = (int64_t)total + (int64_t)rank * bd + tid; i < a.k; i += (int64_t)C * bd) {
            oi[i] = -1;
            if (ov) ov[i] = -INFINITY;
        }
    }
    pdl_trigger();
    // no CTA touches another's shared memory after its last barrier: each may leave now
}

// Counts of the first radix digit of the visible block maxima (a CTA per chunk of a
// row, atomics into the zeroed row histogram).
constexpr int HIST_CHUNK = 8192;

__global__ void __launch_bounds__(256) block_hist_zero_kernel(uint32_t* hist, int64_t words) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i * 4 < words) reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(256) block_hist_kernel(const float* bmax, int64_t ld, const int64_t* nv, int block,
                                                         uint32_t* hist) {
    __shared__ uint32_t h[NB_A];
    pdl_wait();
    const int64_t row = blockIdx.y;
    const int64_t V = nv[row];
    const int64_t nb = min(ld, V > 0 ? (V + block - 1) / block : (int64_t)0);
    const int64_t c0 = (int64_t)blockIdx.x * HIST_CHUNK, c1 = min(nb, c0 + HIST_CHUNK);
    for (int i = threadIdx.x; i < NB_A; i += 256) h[i] = 0u;
    __syncthreads();
    for (int64_t i = c0 + threadIdx.x; i < c1; i += 256) atomicAdd(&h[order_key(bmax[row * ld + i]) >> 20], 1u);
    __syncthreads();
    pdl_trigger();
    if (c0 >= c1) return;
    for (int i = threadIdx.x; i < NB_A; i += 256)
        if (h[i]) atomicAdd(&hist[row * NB_A + i], h[i]);
}

int pool_cluster_size(const csa2_ctx* ctx, int64_t rows, int64_t ld) {
    for (int c : {8, 16, 4, 2, 1}) {
        if (((ld + c - 1) / c + CL_THREADS - 1) / CL_THREADS * CL_THREADS > CL_MAX_CHUNK) continue;
        if (c > 1 && rows * c > ctx->num_sms) continue;
        return c;
    }
    return 16;
}

size_t pool_hist_smem(int chunk, bool entry, int dense_cap = 2 * PH_CAP) {
    const int skey_words = entry ? std::max(chunk, 2 * PH_ECAP) : chunk;
    return (size_t)skey_words * 4 + (size_t)chunk / 32 * 16 + (2ull * PH_CAP + (entry ? dense_cap : 2 * PH_CAP)) * 8;
}

// Whether 16-CTA clusters of the pool kernel can be resident (asked once).
template <bool ENTRY>
bool pool_cluster16_ok() {
    static int ok = -1;
    if (ok < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(CL_THREADS, 1, 1);
        cfg.dynamicSmemBytes = pool_hist_smem(CL_MAX_CHUNK, ENTRY, PH_ECAP);
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 16;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        ok = cudaOccupancyMaxActiveClusters(&n, pool_hist_kernel<ENTRY>, &cfg) == cudaSuccess && n > 0;
        (void)cudaGetLastError();
    }
    return ok == 1;
}

template <bool ENTRY>
csa2_status launch_pool_hist(csa2_ctx* ctx, const PoolArgs& a, int64_t rows, cudaStream_t s) {
    int C = pool_cluster_size(ctx, rows, a.ld);
    auto kern = pool_hist_kernel<ENTRY>;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)pool_hist_smem(CL_MAX_CHUNK, ENTRY, PH_ECAP)) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return CSA2_ERR_CUDA;
        attr = true;
    }
    if (C == 16 && !pool_cluster16_ok<ENTRY>()) C = 8;
    const int chunk = (int)(((a.ld + C - 1) / C + CL_THREADS - 1) / CL_THREADS * CL_THREADS);
    if (chunk > CL_MAX_CHUNK) return CSA2_ERR_UNSUPPORTED;
    // ENTRY: the bitmap of a chunk's entries lives in the candidate lists' space
    if (ENTRY && ((size_t)chunk * a.block + 31) / 32 * 4 > 2ull * PH_CAP * 8) return CSA2_ERR_UNSUPPORTED;
    const size_t smem = pool_hist_smem(chunk, ENTRY, ENTRY ? ph_dense_cap(a.k, a.block) : 2 * PH_CAP);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)rows, 1);
    cfg.blockDim = dim3(CL_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, a, chunk) != cudaSuccess) return CSA2_ERR_CUDA;
    return csa2_launch_status();
}

template <int MODE>
csa2_status run_select(csa2_ctx* ctx, SelArgs a, int64_t rows, int64_t n_max, void* ws, size_t ws_bytes,
                       cudaStream_t s) {
    if (const int C = cluster_size_for(ctx, rows, n_max)) {
        if (ctx->cluster16 < 0) {
            // can a 16-CTA cluster of this kernel be resident at all?
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16, 1, 1);
            cfg.blockDim = dim3(CL_THREADS, 1, 1);                 // the largest block the path launches
            cfg.dynamicSmemBytes = CL_MAX_CHUNK * sizeof(uint32_t);
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 16;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int ncl = 0;
            cudaFuncSetAttribute(sel_cluster_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CL_MAX_CHUNK * 4);
            cudaFuncSetAttribute(sel_cluster_kernel<MODE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            const bool ok = cudaOccupancyMaxActiveClusters(&ncl, sel_cluster_kernel<MODE>, &cfg) == cudaSuccess &&
                            ncl > 0;
            (void)cudaGetLastError();
            ctx->cluster16 = ok ? 1 : 0;
        }
        const int Cuse = (C == 16 && !ctx->cluster16) ? 8 : C;
        if (((n_max + Cuse - 1) / Cuse + 31) / 32 * 32 <= CL_MAX_CHUNK && rows * Cuse <= ctx->num_sms)
            return launch_cluster<MODE>(ctx, a, rows, n_max, Cuse, s);
    }
    bool smem = false;
    choose_chunks(ctx, rows, n_max, a.k, ws_bytes, ws != nullptr, a.chunks, a.chunk_len, smem);
    if (a.chunks > 1) {
        a.ws_key = reinterpret_cast<uint32_t*>(ws);
        a.ws_id = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) +
                                             (size_t)rows * a.chunks * a.k * sizeof(uint32_t));
    } else {
        a.ws_key = nullptr;
        a.ws_id = nullptr;
    }
    static bool attr = false;
    if (!attr) {
        const int bytes = (SEL_SMEM_CAP + 32 + CAND_CAP) * (int)sizeof(uint32_t);
        if (cudaFuncSetAttribute(sel_chunk_kernel<MODE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
                cudaSuccess ||
            cudaFuncSetAttribute(sel_chunk_kernel<MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CAND_CAP * (int)sizeof(uint32_t)) != cudaSuccess ||
            cudaFuncSetAttribute(sel_merge_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
                cudaSuccess)
            return CSA2_ERR_CUDA;
        attr = true;
    }
    if (MODE == SEL_TOPK && a.chunks == 1 && smem && rows >= 2LL * ctx->num_sms && n_max <= SEL_SMEM_CAP &&
        (a.ld % 4) == 0 && aligned(a.vals, 16)) {
        static bool sattr = false;
        if (!sattr) {
            if (cudaFuncSetAttribute(sel_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     CAND_CAP * (int)sizeof(uint32_t)) != cudaSuccess)
                return CSA2_ERR_CUDA;
            sattr = true;
        }
        sel_stream_kernel<<<(unsigned)rows, STREAM_THREADS, CAND_CAP * sizeof(uint32_t), s>>>(a);
        return csa2_launch_status();
    }
    dim3 grid((unsigned)a.chunks, (unsigned)rows);
    if (smem)
        sel_chunk_kernel<MODE, true><<<grid, SEL_THREADS, ((a.chunk_len + 31) / 32 * 32 + CAND_CAP) *
                                                                   sizeof(uint32_t), s>>>(a);
    else
        sel_chunk_kernel<MODE, false><<<grid, SEL_THREADS, CAND_CAP * sizeof(uint32_t), s>>>(a);
    if (a.chunks > 1)
        sel_merge_kernel<MODE><<<(unsigned)rows, SEL_THREADS,
                                 (((size_t)a.chunks * a.k + 31) / 32 * 32 + CAND_CAP) * sizeof(uint32_t), s>>>(a);
    return csa2_launch_status();
}

size_t select_ws_bytes(csa2_ctx* ctx, int64_t rows, int64_t n_max, int k) {
    int chunks = 1;
    int64_t len = 0;
    bool smem = false;
    choose_chunks(ctx, rows, n_max, k, SIZE_MAX / 4, true, chunks, len, smem);
    if (chunks <= 1) return 0;
    return (size_t)rows * chunks * k * (sizeof(uint32_t) + sizeof(int32_t));
}

}  // namespace

extern "C" size_t csa2_topk_workspace_bytes(csa2_ctx* ctx, int64_t rows, int64_t n, int k) {
    if (!ctx || rows <= 0 || n <= 0 || k < 1 || rows > 65535) return 0;
    return select_ws_bytes(ctx, rows, n, k);
}

// The workspace of csa2_block_pool: the row histograms when the caller passes none,
// or the general path's chunk winners, whichever is larger.
extern "C" size_t csa2_block_pool_workspace_bytes(csa2_ctx* ctx, int64_t rows, int64_t ld, int n_keep) {
    if (!ctx || rows <= 0 || ld <= 0 || n_keep < 2 || rows > 65535) return 0;
    return std::max(select_ws_bytes(ctx, rows, ld, n_keep - 1), (size_t)rows * NB_A * sizeof(uint32_t));
}

extern "C" csa2_status csa2_topk(csa2_ctx* ctx, const float* scores, int64_t rows, int64_t n, int64_t ld,
                                 const int64_t* n_visible, const int32_t* pool_blocks, int n_pool, int block,
                                 int k, int32_t* out_idx, float* out_score, void* ws, size_t ws_bytes,
                                 void* stream) {
    if (!ctx || rows < 0 || n < 0 || k < 1 || k > 4096) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
    if (!scores || !n_visible || !out_idx || !aligned(ws, 16)) return CSA2_ERR_INVALID_ARG;
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
        return run_select<SEL_CAND>(ctx, a, rows, a.n, ws, ws_bytes, s);
    }
    if (ld < n) return CSA2_ERR_INVALID_ARG;
    a.n = n;
    return run_select<SEL_TOPK>(ctx, a, rows, n, ws, ws_bytes, s);
}

extern "C" csa2_status csa2_block_pool(csa2_ctx* ctx, const float* block_max, const uint32_t* block_hist,
                                       int64_t rows, int64_t ld, const int64_t* n_visible, int block, int n_keep,
                                       int32_t* out_blocks, int32_t* out_top, int n_top, void* ws,
                                       size_t ws_bytes, void* stream) {
    if (!ctx || rows < 0 || ld < 0 || block < 1 || n_keep < 1 || n_keep > 4096) return CSA2_ERR_INVALID_ARG;
    if (n_top < 0 || n_top > 4096 || (n_top > 0 && !out_top)) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
    if (!block_max || !n_visible || !out_blocks || !aligned(ws, 16) || !aligned(block_hist, 16))
        return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    // with the row histograms (given, or built here in the workspace) the selection
    // reads the maxima once; without them the general radix select runs
    const uint32_t* hist = block_hist;
    const size_t hbytes = (size_t)rows * NB_A * sizeof(uint32_t);
    const bool fits = ld > 0 && ((ld + PH_MAX_C - 1) / PH_MAX_C + CL_THREADS - 1) / CL_THREADS * CL_THREADS <= CL_MAX_CHUNK;
    if (!hist && fits && ws && ws_bytes >= hbytes) {
        uint32_t* h = reinterpret_cast<uint32_t*>(ws);
        csa2_status r = block_hist_zero(h, rows, s);
        if (r == CSA2_OK) r = block_hist_from_max(block_max, rows, ld, n_visible, block, h, s);
        if (r != CSA2_OK) return r;
        hist = h;
    }
    if (hist && fits && n_keep >= 2) {
        PoolArgs p;
        p.bmax = block_max;
        p.ld = ld;
        p.nv = n_visible;
        p.hist = hist;
        p.block = block;
        p.n_keep = n_keep;
        p.out_pool = out_blocks;
        p.n_top = n_top;
        p.out_top = n_top > 0 ? out_top : nullptr;
        p.st = ctx->status;
        p.scores = nullptr;
        p.n_ent = 0;
        p.k = 0;
        p.out_idx = nullptr;
        p.out_val = nullptr;
        return launch_pool_hist<false>(ctx, p, rows, s);
    }
    if (n_top > 0) return CSA2_ERR_UNSUPPORTED;   // the top blocks need a histogram
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
    return run_select<SEL_POOL>(ctx, a, rows, ld, ws, ws_bytes, s);
}

extern "C" csa2_status csa2_pool_topk(csa2_ctx* ctx, const float* block_max, const uint32_t* block_hist,
                                      const float* scores, int64_t rows, int64_t ld, int64_t n_ent,
                                      const int64_t* n_visible, int block, int n_keep, int k, int32_t* out_blocks,
                                      int32_t* out_idx, float* out_score, void* stream) {
    if (!ctx || rows < 0 || ld < 0 || block < 1 || block > 32 || n_keep < 2 || n_keep > 4096 || k < 1)
        return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
    if (!block_max || !block_hist || !scores || !n_visible || !out_blocks || !out_idx || ld <= 0 ||
        n_ent < ld * block || !aligned(block_hist, 16))
        return CSA2_ERR_INVALID_ARG;
    // every entry of the k best blocks is pushed to every CTA of the row's cluster and
    // may be a candidate: they must fit the receive buffer and the candidate list
    if ((int64_t)k * block > PH_ECAP || k > n_keep - 1) return CSA2_ERR_UNSUPPORTED;
    if (((ld + PH_MAX_C - 1) / PH_MAX_C + CL_THREADS - 1) / CL_THREADS * CL_THREADS > CL_MAX_CHUNK)
        return CSA2_ERR_UNSUPPORTED;
    PoolArgs p;
    p.bmax = block_max;
    p.ld = ld;
    p.nv = n_visible;
    p.hist = block_hist;
    p.block = block;
    p.n_keep = n_keep;
    p.out_pool = out_blocks;
    p.n_top = k;
    p.out_top = nullptr;
    p.st = ctx->status;
    p.scores = scores;
    p.n_ent = n_ent;
    p.k = k;
    p.out_idx = out_idx;
    p.out_val = out_score;
    return launch_pool_hist<true>(ctx, p, rows, as_stream(stream));
}

extern "C" csa2_status csa2_block_hist(csa2_ctx* ctx, const float* block_max, int64_t rows, int64_t ld,
                                       const int64_t* n_visible, int block, uint32_t* block_hist, void* stream) {
    if (!ctx || rows < 0 || ld < 0 || block < 1) return CSA2_ERR_INVALID_ARG;
    if (rows == 0) return CSA2_OK;
    if (rows > 65535) return CSA2_ERR_UNSUPPORTED;
    if (!block_max || !n_visible || !block_hist || !aligned(block_hist, 16)) return CSA2_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    const csa2_status r = block_hist_zero(block_hist, rows, s);
    return r != CSA2_OK ? r : block_hist_from_max(block_max, rows, ld, n_visible, block, block_hist, s);
}

csa2_status block_hist_zero(uint32_t* hist, int64_t rows, cudaStream_t s) {
    const int64_t words = rows * NB_A;
    const csa2_status r = launch_pdl(block_hist_zero_kernel, dim3((unsigned)((words / 4 + 255) / 256)), dim3(256), 0,
                                     s, hist, words);
    return r != CSA2_OK ? r : csa2_launch_status();
}

csa2_status block_hist_from_max(const float* bmax, int64_t rows, int64_t ld, const int64_t* n_visible, int block,
                                uint32_t* hist, cudaStream_t s) {
    if (ld <= 0) return CSA2_OK;
    const csa2_status r = launch_pdl(block_hist_kernel, dim3((unsigned)((ld + HIST_CHUNK - 1) / HIST_CHUNK), (unsigned)rows),
                                     dim3(256), 0, s, bmax, ld, n_visible, block, hist);
    return r != CSA2_OK ? r : csa2_launch_status();
}
