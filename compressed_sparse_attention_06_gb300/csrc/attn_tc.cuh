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
// row many times over, the rows' RMS factors (B*N + B*swa_cap floats).  More than 64
// heads run in passes of 64 that reuse the workspace, so H is capped at 64 here.
// The path runs with any workspace that holds the partials and the images.
size_t attn_tc_ws_bytes(const csa2_ctx* ctx, int B, int Q, int H, int k, int window, int64_t N, int64_t swa_cap);

// Workspace bytes of the CUDA-core path (attn.cu) for these sizes: its key-split
// partials, 0 when it runs unsplit.
size_t attn_simt_ws_bytes(const csa2_ctx* ctx, int B, int Q, int H, int k, int window);

// The RoPE cos/sin table (float [B*Q, 64]) the path wrote into `ws` for this call.
const float* attn_tc_rope_table(const csa2_ctx* ctx, const AttnTcCall& c, void* ws);

// Runs the path.  On return *n_split > 1 means the output is still in per-split
// partials at the start of `ws` (float [B*Q, H, n_split, ATTN_PART]),
// to be merged by the caller's combine kernel.
csa2_status attn_tc_run(csa2_ctx* ctx, const AttnTcCall& c, void* ws, size_t ws_bytes, cudaStream_t s,
                        int* n_split);
