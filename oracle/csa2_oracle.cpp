// CPU oracle for the CSA2 compressed-sparse-attention hot path, in plain C++17.
//
// TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the bench's
// CPU-baseline / reference leg may load or run this library.  It shares no code,
// header, table or constant generator with the CUDA library; it restates the same
// definitions as the numpy oracle (oracle/csa2_oracle.py), in double precision,
// with plain loops and the standard library only.  The tests hold the two oracles to
// each other on the pinned examples and on random inputs.
//
// Sources (three web pages on CSA / CSA2), cited by short title:
//   "CSA2 page"                 «CSA2：跨层共享的压缩稀疏注意力»
//   "Attention-evolution page"  «DeepSeek 的 Attention 演进 -【DSA、CSA、CSA2】»
//   "DSA-to-CSA/HCA page"       «从 DSA 到 CSA/HCA：先压缩时间轴，再决定怎样寻址»
//
// Readings where the pages are silent are the numpy oracle's (its header lists
// them): no indexer scale; t >= m(j+1) visibility; lower index wins a top-k tie;
// the newest visible block always in the pool; RMSNorm eps 1e-6 with unit gain;
// RoPE on the last 64 dims as interleaved pairs, base 10000, angle in double reduced
// mod 2 pi; FP4 scales E4M3_RNE(f32(amax)/6), MXFP4 scales 2^(floor(log2 amax)-2).
//
// The one parallel part is the driver of the decode baseline: the indexer scan over
// the entries is split into contiguous ranges, one per std::thread.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <thread>
#include <vector>

namespace {

const double NEG_INF = -std::numeric_limits<double>::infinity();
const double TWO_PI = 6.283185307179586476925286766559;
constexpr int ROPE_DIMS = 64;
constexpr double RMS_EPS = 1e-6;
enum { QNORM = 1, KVNORM = 2, ROPE = 4 };
enum { NORM_W = 1, ROPE_W = 2 };

// ---------------------------------------------------------------- minifloats (OCP)
// sign / exponent / mantissa fields to a value; no inf or NaN handling here
double minifloat(int code, int ebits, int mbits, int bias) {
    const int m = code & ((1 << mbits) - 1);
    const int e = (code >> mbits) & ((1 << ebits) - 1);
    const int s = (code >> (mbits + ebits)) & 1;
    const double frac = (double)m / (double)(1 << mbits);
    const double mag = e > 0 ? std::ldexp(1.0 + frac, e - bias) : std::ldexp(frac, 1 - bias);
    return s ? -mag : mag;
}

double e2m1_value(int code) { return minifloat(code & 0xF, 2, 1, 1); }
double e4m3_value(int code) {
    if ((code & 0x7F) == 0x7F) return std::numeric_limits<double>::quiet_NaN();
    return minifloat(code & 0xFF, 4, 3, 7);
}
double e8m0_value(int code) {
    if (code == 0xFF) return std::numeric_limits<double>::quiet_NaN();
    return std::ldexp(1.0, code - 127);
}

// Nearest grid value to |x| (grid ascending from 0, saturating at its top), ties to
// the code with a 0 mantissa lsb (round to nearest even); returns the magnitude code.
int rne_code(double x, const std::vector<double>& grid) {
    double a = std::fabs(x);
    a = std::min(a, grid.back());
    size_t hi = std::lower_bound(grid.begin(), grid.end(), a) - grid.begin();
    hi = std::min(hi, grid.size() - 1);
    const size_t lo = hi > 0 ? hi - 1 : 0;
    const double dlo = a - grid[lo], dhi = grid[hi] - a;
    if (dhi < dlo) return (int)hi;
    if (dhi > dlo) return (int)lo;
    return (hi & 1) == 0 ? (int)hi : (int)lo;
}

const std::vector<double>& e2m1_grid() {
    static const std::vector<double> g = [] {
        std::vector<double> v;
        for (int c = 0; c < 8; ++c) v.push_back(e2m1_value(c));
        return v;
    }();
    return g;
}
const std::vector<double>& e4m3_grid() {
    static const std::vector<double> g = [] {
        std::vector<double> v;
        for (int c = 0; c < 0x7F; ++c) v.push_back(e4m3_value(c));
        return v;
    }();
    return g;
}

int e2m1_encode(double x) { return rne_code(x, e2m1_grid()) | (std::signbit(x) ? 8 : 0); }
int e4m3_encode(double x) { return rne_code(x, e4m3_grid()) | (std::signbit(x) ? 0x80 : 0); }

// ---------------------------------------------------------------- RMSNorm, RoPE
void rms_norm(double* x, int c) {
    double ss = 0.0;
    for (int i = 0; i < c; ++i) ss += x[i] * x[i];
    const double r = std::sqrt(ss / c + RMS_EPS);
    for (int i = 0; i < c; ++i) x[i] /= r;
}

// Rotate the last 64 dims of x (pairs (c-64+2j, c-63+2j)) by +pos, or by -pos.
void rope(double* x, int c, int64_t pos, bool inverse, double base) {
    for (int j = 0; j < ROPE_DIMS / 2; ++j) {
        const double theta = std::pow(base, -2.0 * j / ROPE_DIMS);
        const double ang = std::fmod((double)pos * theta, TWO_PI);
        const double cs = std::cos(ang), sn = inverse ? -std::sin(ang) : std::sin(ang);
        double& x0 = x[c - ROPE_DIMS + 2 * j];
        double& x1 = x[c - ROPE_DIMS + 2 * j + 1];
        const double a = x0, b = x1;
        x0 = a * cs - b * sn;
        x1 = a * sn + b * cs;
    }
}

// ---------------------------------------------------------------- selection order
// (value desc, index asc): the one total order of every selection.
struct ByValueThenIndex {
    const double* v;
    bool operator()(int64_t a, int64_t b) const {
        if (v[a] != v[b]) return v[a] > v[b];
        return a < b;
    }
};

}  // namespace

extern "C" {

int csa2o_version() { return 1; }

// ---------------------------------------------------------------- FP4 formats
// (CSA2 page, «890 字节是怎么来的»: FP4 main KV 288 B, MXFP4 indexer K 68 B)
double csa2o_e2m1_value(int code) { return e2m1_value(code); }
double csa2o_e4m3_value(int code) { return e4m3_value(code); }
double csa2o_e8m0_value(int code) { return e8m0_value(code); }
int csa2o_e2m1_encode(double x) { return e2m1_encode(x); }
int csa2o_e4m3_encode(double x) { return e4m3_encode(x); }

// FP4 main-KV rows: per 16 channels s = E4M3_RNE(f32(amax) / 6) (f32 division),
// s == 0 -> all codes 0, else code = E2M1_RNE(f32(x) / s) (f32 division); channel 2i
// in the low nibble; a row is c/2 code bytes then c/16 scale bytes.
void csa2o_nvfp4_pack(const float* x, int64_t rows, int c, uint8_t* out) {
    const int rb = c / 2 + c / 16;
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * c;
        uint8_t* o = out + r * rb;
        for (int g = 0; g < c / 16; ++g) {
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(xr[16 * g + i]));
            const float s32 = amax / 6.0f;
            const int scode = e4m3_encode((double)s32);
            const float sval = (float)e4m3_value(scode);
            o[c / 2 + g] = (uint8_t)scode;
            for (int i = 0; i < 16; i += 2) {
                int lo = 0, hi = 0;
                if (sval != 0.0f) {
                    lo = e2m1_encode((double)(xr[16 * g + i] / sval));
                    hi = e2m1_encode((double)(xr[16 * g + i + 1] / sval));
                }
                o[(16 * g + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

void csa2o_nvfp4_unpack(const uint8_t* in, int64_t rows, int c, double* out) {
    const int rb = c / 2 + c / 16;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* b = in + r * rb;
        for (int i = 0; i < c; ++i) {
            const int code = (b[i / 2] >> (4 * (i & 1))) & 0xF;
            out[r * c + i] = e2m1_value(code) * e4m3_value(b[c / 2 + i / 16]);
        }
    }
}

// MXFP4 rows (OCP MX): per 32 values X = 2^(floor(log2 amax) - 2) as E8M0 clamped to
// [0, 254]; amax == 0 -> scale byte 0 and codes 0; code = E2M1_RNE(f32(x) / X); a
// row is d/2 code bytes then d/32 scale bytes.
void csa2o_mxfp4_pack(const float* x, int64_t rows, int d, uint8_t* out) {
    const int rb = d / 2 + d / 32;
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * d;
        uint8_t* o = out + r * rb;
        for (int g = 0; g < d / 32; ++g) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(xr[32 * g + i]));
            int code = 0;
            if (amax != 0.0f) {
                int ex = 0;
                std::frexp((double)amax, &ex);               // amax = f 2^ex, f in [0.5, 1)
                code = std::min(254, std::max(0, ex - 1 - 2 + 127));
            }
            o[d / 2 + g] = (uint8_t)code;
            const float X = (float)e8m0_value(code);
            for (int i = 0; i < 32; i += 2) {
                int lo = 0, hi = 0;
                if (amax != 0.0f) {
                    lo = e2m1_encode((double)(xr[32 * g + i] / X));
                    hi = e2m1_encode((double)(xr[32 * g + i + 1] / X));
                }
                o[(32 * g + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

void csa2o_mxfp4_unpack(const uint8_t* in, int64_t rows, int d, double* out) {
    const int rb = d / 2 + d / 32;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* b = in + r * rb;
        for (int i = 0; i < d; ++i) {
            const int code = (b[i / 2] >> (4 * (i & 1))) & 0xF;
            out[r * d + i] = e2m1_value(code) * e8m0_value(b[d / 2 + i / 32]);
        }
    }
}

// ---------------------------------------------------------------- compressor
// Non-overlapping form (Attention-evolution page §4.1; DSA-to-CSA/HCA page eqs.
// (22)-(23)): per channel a softmax over the m positions of block i of Z^a + B^a,
// E[i] = sum_j S_j C^a_j.  Overlapping form (DSA-to-CSA/HCA page eqs. (11)-(12)), when
// Cb is given: the softmax runs over the 2m rows [Z^a_cur + B^a ; Z^b_prev + B^b],
// weighting [C^a_cur ; C^b_prev]; the first block's history is (prev_Cb, prev_Zb) or
// (0, -inf).  Ba, Bb may be NULL (0).  Shapes: C*, Z* [n, c]; B*, prev_* [m, c].
void csa2o_compress(const double* Ca, const double* Za, int64_t n, int c, int m, const double* Ba, const double* Cb,
                    const double* Zb, const double* Bb, const double* prev_Cb, const double* prev_Zb, double* out) {
    const bool overlap = Cb != nullptr;
    std::vector<double> pC((size_t)m * c, 0.0), pZ((size_t)m * c, NEG_INF);
    if (overlap && prev_Cb) std::copy(prev_Cb, prev_Cb + (size_t)m * c, pC.begin());
    if (overlap && prev_Zb) std::copy(prev_Zb, prev_Zb + (size_t)m * c, pZ.begin());
    std::vector<double> lg(2 * m), val(2 * m);
    for (int64_t i = 0; i < n / m; ++i) {
        for (int ch = 0; ch < c; ++ch) {
            int rows = 0;
            for (int j = 0; j < m; ++j) {
                const int64_t t = i * m + j;
                lg[rows] = Za[t * c + ch] + (Ba ? Ba[(size_t)j * c + ch] : 0.0);
                val[rows] = Ca[t * c + ch];
                ++rows;
            }
            if (overlap) {
                for (int j = 0; j < m; ++j) {
                    lg[rows] = pZ[(size_t)j * c + ch] + (Bb ? Bb[(size_t)j * c + ch] : 0.0);
                    val[rows] = pC[(size_t)j * c + ch];
                    ++rows;
                }
            }
            double mx = NEG_INF;
            for (int r = 0; r < rows; ++r) mx = std::max(mx, lg[r]);
            double den = 0.0, num = 0.0;
            for (int r = 0; r < rows; ++r) {
                const double e = std::exp(lg[r] - mx);
                den += e;
                num += e * val[r];
            }
            out[i * c + ch] = num / den;
        }
        if (overlap) {
            for (int j = 0; j < m; ++j)
                for (int ch = 0; ch < c; ++ch) {
                    pC[(size_t)j * c + ch] = Cb[(i * m + j) * c + ch];
                    pZ[(size_t)j * c + ch] = Zb[(i * m + j) * c + ch];
                }
        }
    }
}

// Write epilogue: [RMSNorm] -> [RoPE of entry i at pos0 + m i], in place on E [ne, c].
void csa2o_compress_write(double* E, int64_t ne, int c, int flags, int m, int64_t pos0, double base) {
    for (int64_t i = 0; i < ne; ++i) {
        if (flags & NORM_W) rms_norm(E + i * c, c);
        if (flags & ROPE_W) rope(E + i * c, c, pos0 + (int64_t)m * i, false, base);
    }
}

void csa2o_rms_norm(double* x, int64_t rows, int c) {
    for (int64_t r = 0; r < rows; ++r) rms_norm(x + r * c, c);
}

void csa2o_rope(double* x, int64_t rows, int c, int64_t pos, int inverse, double base) {
    for (int64_t r = 0; r < rows; ++r) rope(x + r * c, c, pos, inverse != 0, base);
}

// ---------------------------------------------------------------- indexer
// I[s] = sum_h w[h] ReLU(q^I_h . K^I_s) for s < V, -inf beyond (DSA-to-CSA/HCA page
// eq. (16): no scale, no softmax).  qI [H, d], w [H], K [N, d].
void csa2o_index_score(const double* qI, const double* w, const double* K, int64_t N, int64_t V, int H, int d,
                       double* out) {
    for (int64_t s = 0; s < N; ++s) {
        if (s >= V) {
            out[s] = NEG_INF;
            continue;
        }
        double acc = 0.0;
        for (int h = 0; h < H; ++h) {
            double dot = 0.0;
            for (int i = 0; i < d; ++i) dot += qI[(size_t)h * d + i] * K[s * d + i];
            acc += w[h] * std::max(dot, 0.0);
        }
        out[s] = acc;
    }
}

// Top-k of the V visible entries by (score desc, index asc); all of them if V <= k;
// ids ascending, -1 padded (DSA-to-CSA/HCA page eq. (17)).
void csa2o_topk(const double* scores, int64_t V, int k, int64_t* out) {
    std::vector<int64_t> ids((size_t)std::max<int64_t>(V, 0));
    std::iota(ids.begin(), ids.end(), 0);
    std::sort(ids.begin(), ids.end(), ByValueThenIndex{scores});
    const int64_t n = std::min<int64_t>(k, V > 0 ? V : 0);
    std::vector<int64_t> sel(ids.begin(), ids.begin() + n);
    std::sort(sel.begin(), sel.end());
    for (int i = 0; i < k; ++i) out[i] = i < n ? sel[i] : -1;
}

// Block score = max over the visible members of each block (CSA2 page,
// «解码器里的分层索引»); ceil(V / block) blocks.
void csa2o_block_max(const double* scores, int64_t V, int block, double* out) {
    const int64_t nb = V > 0 ? (V + block - 1) / block : 0;
    for (int64_t b = 0; b < nb; ++b) {
        double m = NEG_INF;
        for (int64_t s = b * block; s < std::min<int64_t>(V, b * block + block); ++s) m = std::max(m, scores[s]);
        out[b] = m;
    }
}

// The pool: the newest visible block floor((V-1)/block) always, the other n_keep-1
// slots to the best other blocks by (block max desc, block asc); every visible block
// if they fit; ascending, -1 padded (CSA2 page, «解码器里的分层索引»).
void csa2o_block_pool(const double* bmax, int64_t V, int block, int n_keep, int64_t* out) {
    for (int i = 0; i < n_keep; ++i) out[i] = -1;
    if (V <= 0) return;
    const int64_t nb = (V + block - 1) / block, b_new = (V - 1) / block;
    if (nb <= n_keep) {
        for (int64_t b = 0; b < nb; ++b) out[b] = b;
        return;
    }
    std::vector<int64_t> others;
    for (int64_t b = 0; b < nb; ++b)
        if (b != b_new) others.push_back(b);
    std::sort(others.begin(), others.end(), ByValueThenIndex{bmax});
    std::vector<int64_t> sel(others.begin(), others.begin() + (n_keep - 1));
    sel.push_back(b_new);
    std::sort(sel.begin(), sel.end());
    for (int i = 0; i < n_keep; ++i) out[i] = sel[i];
}

// Reindex selection in the official minimal form (Attention-evolution page §4.4): the
// full scores, a mask of the pooled candidates (visible entries of the pool's blocks),
// then the top-k among them by (score desc, index asc); ascending, -1 padded.
void csa2o_reindex_topk(const double* full_scores, const int64_t* pool, int n_pool, int64_t V, int k, int block,
                        int64_t* out) {
    std::vector<int64_t> cand;
    for (int i = 0; i < n_pool; ++i) {
        if (pool[i] < 0) continue;
        for (int r = 0; r < block; ++r) {
            const int64_t s = pool[i] * block + r;
            if (s < V) cand.push_back(s);
        }
    }
    std::sort(cand.begin(), cand.end(), ByValueThenIndex{full_scores});
    const int64_t n = std::min<int64_t>(k, (int64_t)cand.size());
    std::vector<int64_t> sel(cand.begin(), cand.begin() + n);
    std::sort(sel.begin(), sel.end());
    for (int i = 0; i < k; ++i) out[i] = i < n ? sel[i] : -1;
}

// ---------------------------------------------------------------- attention
// One query over given key/value rows, all heads (DSA-to-CSA/HCA page eqs. (18)-(19),
// (27)): q^ = RoPE_t(RMSNorm(q)); k^_j = RMSNorm(row_j); z_j = q^.k^_j / sqrt(c);
// p_j = e^{z_j} / (sum_l e^{z_l} + e^{sink_h}); o = RoPE_-t(sum_j p_j k^_j);
// lse = log(sum_j e^{z_j} + e^{sink_h}).  sink NULL: no sink term.  q [H, c],
// keys [nk, c]; out [H, c], lse [H] (may be NULL).
void csa2o_attend(const double* q, const double* keys, int64_t nk, int H, int c, int64_t t, const double* sink,
                  int flags, double base, double* out, double* lse) {
    std::vector<double> K(keys, keys + nk * c);
    if (flags & KVNORM)
        for (int64_t j = 0; j < nk; ++j) rms_norm(K.data() + j * c, c);
    std::vector<double> qh((size_t)c), z((size_t)std::max<int64_t>(nk, 1));
    for (int h = 0; h < H; ++h) {
        std::copy(q + (size_t)h * c, q + (size_t)(h + 1) * c, qh.begin());
        if (flags & QNORM) rms_norm(qh.data(), c);
        if (flags & ROPE) rope(qh.data(), c, t, false, base);
        double mx = sink ? sink[h] : NEG_INF;
        for (int64_t j = 0; j < nk; ++j) {
            double dot = 0.0;
            for (int i = 0; i < c; ++i) dot += qh[i] * K[j * c + i];
            z[j] = dot / std::sqrt((double)c);
            mx = std::max(mx, z[j]);
        }
        double den = sink ? std::exp(sink[h] - mx) : 0.0;
        for (int64_t j = 0; j < nk; ++j) den += std::exp(z[j] - mx);
        double* o = out + (size_t)h * c;
        for (int i = 0; i < c; ++i) o[i] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            const double p = std::exp(z[j] - mx) / den;
            for (int i = 0; i < c; ++i) o[i] += p * K[j * c + i];
        }
        if (flags & ROPE) rope(o, c, t, true, base);
        if (lse) lse[h] = mx + std::log(den);
    }
}

// The rows of query t: the selected entries (id -1 skipped) then the window rows at
// positions max(0, t-window+1) .. t (slot (p - swa_pos0) mod swa_cap), then attend.
// kv [N, c] entries; idx [k]; swa [swa_cap, c].
void csa2o_sparse_attn(const double* q, const double* kv, const int64_t* idx, int k, const double* swa,
                       int64_t swa_cap, int64_t swa_pos0, int64_t t, const double* sink, int window, int H, int c,
                       int flags, double base, double* out, double* lse) {
    std::vector<double> rows;
    for (int i = 0; i < k; ++i)
        if (idx[i] >= 0) rows.insert(rows.end(), kv + idx[i] * c, kv + (idx[i] + 1) * c);
    if (window > 0)
        for (int64_t p = std::max<int64_t>(0, t - window + 1); p <= t; ++p) {
            const int64_t slot = (((p - swa_pos0) % swa_cap) + swa_cap) % swa_cap;
            rows.insert(rows.end(), swa + slot * c, swa + (slot + 1) * c);
        }
    csa2o_attend(q, rows.data(), (int64_t)rows.size() / c, H, c, t, sink, flags, base, out, lse);
}

// ---------------------------------------------------------------- decode baseline
// One Full-mode decode query over FP4 caches, the steps of the numpy oracle's decode
// sample: dequantise the MXFP4 indexer rows, score every visible entry (one range of
// entries per std::thread), block maxima, pool, top-k inside the pool (the official
// minimal form), dequantise the selected FP4 main-KV rows and attend with the window.
//   ki [N, 68] MXFP4 rows; qI_mx [H_I, 68] the packed indexer query; w [H_I];
//   kv_ids [n_kv] ascending ids with kv_rows [n_kv, 288] their FP4 main-KV rows (at
//   least every selected id); q [H, 512]; swa [swa_cap, 512]; sink [H] or NULL.
//   out [H, 512], lse [H], idx_out [k].
int csa2o_decode_query_fp4(const uint8_t* ki, int64_t N, int64_t V, const uint8_t* qI_mx, const double* w, int H_I,
                           int block, int n_keep, int k, const int64_t* kv_ids, const uint8_t* kv_rows, int64_t n_kv,
                           const double* q, int H, const double* swa, int64_t swa_cap, int64_t swa_pos0, int64_t t,
                           const double* sink, int window, double base, int threads, double* out, double* lse,
                           int64_t* idx_out) {
    const int d = 128, c = 512;
    std::vector<double> qI((size_t)H_I * d);
    csa2o_mxfp4_unpack(qI_mx, H_I, d, qI.data());
    std::vector<double> scores((size_t)std::max<int64_t>(N, 1), NEG_INF);
    const int nt = std::max(1, threads);
    const int64_t Vc = std::min(V, N);
    std::vector<std::thread> pool;
    for (int ti = 0; ti < nt; ++ti) {
        pool.emplace_back([&, ti] {
            const int64_t s0 = Vc * ti / nt, s1 = Vc * (ti + 1) / nt;
            std::vector<double> row(d);
            for (int64_t s = s0; s < s1; ++s) {
                csa2o_mxfp4_unpack(ki + s * (d / 2 + d / 32), 1, d, row.data());
                csa2o_index_score(qI.data(), w, row.data(), 1, 1, H_I, d, &scores[s]);
            }
        });
    }
    for (auto& th : pool) th.join();
    const int64_t nb = Vc > 0 ? (Vc + block - 1) / block : 0;
    std::vector<double> bm((size_t)std::max<int64_t>(nb, 1));
    csa2o_block_max(scores.data(), Vc, block, bm.data());
    std::vector<int64_t> pl((size_t)n_keep);
    csa2o_block_pool(bm.data(), Vc, block, n_keep, pl.data());
    csa2o_reindex_topk(scores.data(), pl.data(), n_keep, Vc, k, block, idx_out);
    // the selected main-KV rows, dequantised, in a dense [k, c] table
    std::vector<double> sel((size_t)k * c, 0.0);
    std::vector<int64_t> local((size_t)k, -1);
    for (int i = 0; i < k; ++i) {
        if (idx_out[i] < 0) continue;
        const int64_t* it = std::lower_bound(kv_ids, kv_ids + n_kv, idx_out[i]);
        if (it == kv_ids + n_kv || *it != idx_out[i]) return 1;   // a selected row was not provided
        csa2o_nvfp4_unpack(kv_rows + (it - kv_ids) * (c / 2 + c / 16), 1, c, sel.data() + (size_t)i * c);
        local[i] = i;
    }
    csa2o_sparse_attn(q, sel.data(), local.data(), k, swa, swa_cap, swa_pos0, t, sink, window, H, c,
                      QNORM | KVNORM | ROPE, base, out, lse);
    return 0;
}

}  // extern "C"
