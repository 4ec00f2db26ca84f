// Tensor-core (tcgen05) path of csa2_sparse_attn, used when the query and the
// window are bf16, the selected rows are bf16 or FP4, both RMSNorms are on and the
// heads fit one 64-wide MMA.  The caller (attn.cu) owns validation and the split
// combine.
#pragma once

#include "csa2_internal.cuh"

// Per-split partial result of one (query, head): [0] = max logit (or the fixed
// offset), [1] = sum of exponentials, [ATTN_PART_O ..] = the 512 unnormalised output
// values.  Rows are 16-byte multiples so they can be written by bulk copies.
constexpr int ATTN_PART = 516;
constexpr int ATTN_PART_O = 4;

// Inverse (sign -1) or forward RoPE on a warp's copy of one 512-dim row, lane l
// holding dims l + 32 i: dims 448..511 are x[14], x[15]; pair (2j, 2j+1) sits in
// lanes (2j, 2j+1) mod 32.  cs / sn: cos / sin of the 32 angles.
__device__ __forceinline__ void rope_lanes(float (&x)[16], int lane, const float* cs, const float* sn, float sign) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int j = (lane + 32 * i) >> 1;
        const float c = cs[j], s = sign * sn[j];
        float v = x[14 + i];
        float p = __shfl_xor_sync(0xffffffffu, v, 1);
        x[14 + i] = (lane & 1) ? fmaf(p, s, v * c) : fmaf(-p, s, v * c);
    }
}

// Merge of the key splits of one (query, head) by one warp (DSA-to-CSA/HCA page eq.
// (27) over the union of the splits' keys): part = the ns partials of the row (max or
// offset, sum of exponentials, unnormalised output), zs = the sink logit (-inf: none),
// cs / sn = RoPE at the query position (NULL: no rotation).  Writes the 512 outputs
// to o and, if lse is not NULL, log(sum e^z + e^zs) to *lse.
template <typename TO>
__device__ __forceinline__ void attn_combine_row(const float* part, int ns, float zs, const float* cs,
                                                 const float* sn, TO* o, float* lse) {
    const int lane = threadIdx.x & 31;
    float M = zs;
    for (int s0 = 0; s0 < ns; s0 += 32)
        M = fmaxf(M, warp_max(s0 + lane < ns ? part[(s0 + lane) * ATTN_PART] : -INFINITY));
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    float denom = 0.0f;
    if (M != -INFINITY) {
        denom = (zs == -INFINITY) ? 0.0f : expf(zs - M);
        for (int s = 0; s < ns; s += 4) {
            float e[4], l[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float ms = s + j < ns ? part[(s + j) * ATTN_PART] : -INFINITY;
                e[j] = (ms == -INFINITY) ? 0.0f : expf(ms - M);
                l[j] = s + j < ns ? part[(s + j) * ATTN_PART + 1] : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (s + j >= ns) break;
                denom = fmaf(l[j], e[j], denom);
                const float* pj = part + (s + j) * ATTN_PART + ATTN_PART_O + lane;
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = fmaf(e[j], pj[32 * i], acc[i]);
            }
        }
    }
    const float inv = denom > 0.0f ? 1.0f / denom : 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= inv;
    if (cs) rope_lanes(acc, lane, cs, sn, -1.0f);
#pragma unroll
    for (int i = 0; i < 16; ++i) o[lane + 32 * i] = from_f32<TO>(acc[i]);
    if (lse && lane == 0) *lse = (denom > 0.0f) ? M + logf(denom) : -INFINITY;
}

struct AttnTcCall {
    const void* q;
    csa2_dtype q_dt;
    const void* kv;
    csa2_dtype kv_dt;
    int64_t N;
    const int32_t* idx;
    int k;                 // idx row length, or (dense_nv) the most entries a query takes
    const int64_t* dense_nv; // dense mode (idx NULL): query bq takes entries 0 .. dense_nv[bq]-1
    const void* swa;
    csa2_dtype swa_dt;
    int64_t swa_cap, swa_pos0;
    int window;
    const int64_t* q_pos;
    const float* sink;
    int B, Q, H;           // H: heads of this pass (<= 64)
    int n_pass = 1;        // > 1: every 64-head pass in one launch (H = 64, q, out, lse and
                           // sink not offset; pass p takes heads 64p .. of Hs)
    int Hs;                // heads per query in q / out / lse (q, out, lse, sink point at this
                           // pass's first head)
    RopeTable rope;
    unsigned flags;
    void* out;
    csa2_dtype out_dt;
    float* lse;
};

// Whether the tensor-core path handles these dtypes, flags and sizes.
bool attn_tc_applies(const AttnTcCall& c);

// Workspace bytes the tensor-core path uses for these sizes: per-split partials
// (when the keys are split), the query images, and, when the call gathers each
// row many times over, the rows' RMS factors (B*N + B*swa_cap floats), for one pass of
// at most 64 heads (H is capped at 64 here; passes run one after another in it).
// The path runs with any workspace that holds the partials and the images.
size_t attn_tc_ws_bytes(const csa2_ctx* ctx, int B, int Q, int H, int k, int window, int64_t N, int64_t swa_cap);

// Workspace bytes of one launch over every head pass of H heads (H > 64): the passes'
// query images and partials side by side.
size_t attn_tc_ws_bytes_all_passes(const csa2_ctx* ctx, int B, int Q, int H, int k, int window, int64_t N,
                                   int64_t swa_cap);

// Workspace bytes of the CUDA-core path (attn.cu) for these sizes: its key-split
// partials, 0 when it runs unsplit.
size_t attn_simt_ws_bytes(const csa2_ctx* ctx, int B, int Q, int H, int k, int window);

// The RoPE cos/sin table (float [B*Q, 64]) the path wrote into `ws` for this call.
const float* attn_tc_rope_table(const csa2_ctx* ctx, const AttnTcCall& c, void* ws);

// The query half of the path alone (query images and RoPE table into `ws`), for a
// later attn_tc_run with CSA2_ATTN_PREPARED in the flags and the same sizes.
csa2_status attn_tc_prepare(csa2_ctx* ctx, const AttnTcCall& c, void* ws, size_t ws_bytes, cudaStream_t s);

// Runs the path.  On return *n_split > 1 means the output is still in per-split
// partials at the start of `ws` (float [B*Q, H, n_split, ATTN_PART]),
// to be merged by the caller's combine kernel.
csa2_status attn_tc_run(csa2_ctx* ctx, const AttnTcCall& c, void* ws, size_t ws_bytes, cudaStream_t s,
                        int* n_split);
