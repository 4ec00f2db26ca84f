/*
 * csa2.h -- C ABI of the CSA2 compressed-sparse-attention hot path (sm_103a).
 *
 * The path (all on one GPU, all in this library's CUDA kernels):
 *   compressor -> [FP4 pack] -> Lightning-indexer scores (+ block max)
 *   -> block pool / top-512 (Full, Reindex) or upstream indices (Reuse)
 *   -> shared-KV MQA over the selected entries plus the sliding window.
 *
 * Sources, cited by short title:
 *   "CSA2 page"                 «CSA2：跨层共享的压缩稀疏注意力» (daiw.org)
 *   "Attention-evolution page"  «DeepSeek 的 Attention 演进 -【DSA、CSA、CSA2】»
 *   "DSA-to-CSA/HCA page"       «从 DSA 到 CSA/HCA：先压缩时间轴，再决定怎样寻址»
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library never
 *     allocates tensors.  All tensors are dense row-major with the shapes given.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Arguments are validated on the host before any launch;
 *     on a validation failure nothing is launched.
 *   - Kernels never trap.  A kernel that meets an out-of-range index skips the
 *     access and records CSA2_ERR_DEVICE in the context's status word; a bounded
 *     wait that expires records CSA2_ERR_TIMEOUT.  csa2_ctx_check() reads (and
 *     clears) that word.
 *   - No call throws, exits or prints.
 *   - A context is used by one host thread at a time.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = 1,   /* bad pointer / size / alignment; nothing launched   */
    CSA2_ERR_UNSUPPORTED = 2,   /* valid, but a dtype/shape combination not provided  */
    CSA2_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed               */
    CSA2_ERR_TIMEOUT = 4,       /* a device-side bounded wait expired (from the ctx)  */
    CSA2_ERR_DEVICE = 5         /* a kernel saw an out-of-range index (from the ctx)  */
} csa2_status;

typedef enum {
    CSA2_F32 = 0,
    CSA2_BF16 = 1,
    /* FP4 main-KV row, 512 channels -> 288 B: 256 B of E2M1 codes (channel 2i in the
       low nibble of byte i) then 32 E4M3 scales, one per 16 channels (CSA2 page,
       «890 字节是怎么来的»).  Rows of other widths c (c % 16 == 0): c/2 + c/16 B. */
    CSA2_FP4_E4M3x16 = 2,
    /* MXFP4 indexer-K row, 128 dims -> 68 B: 64 B of E2M1 codes then 4 E8M0 scales,
       one per 32 values (same section).  Width d (d % 32 == 0): d/2 + d/32 B.        */
    CSA2_MXFP4_E8M0x32 = 3
} csa2_dtype;

/* attention flags */
#define CSA2_QNORM  1u   /* RMSNorm each query head before attention              */
#define CSA2_KVNORM 2u   /* RMSNorm each key/value row (compressed and window)    */
#define CSA2_ROPE   4u   /* RoPE_t on the query's last 64 dims, RoPE_-t on output */
#define CSA2_ATTN_DEFAULT (CSA2_QNORM | CSA2_KVNORM | CSA2_ROPE)
#define CSA2_ATTN_PREPARED 8u  /* csa2_attn_prepare already wrote the query half into ws */

/* compressor write-epilogue flags */
#define CSA2_W_NORM 1u   /* RMSNorm of each compressed entry (kv_norm)            */
#define CSA2_W_ROPE 2u   /* RoPE of the entry's last 64 dims at position pos0+m*i */

typedef struct csa2_ctx csa2_ctx;

const char* csa2_status_string(csa2_status s);
int csa2_version(void);

/* Create a context on `device`: it holds a 4-byte device status word (the only
   allocation this library makes) and the device's SM count. */
csa2_status csa2_ctx_create(int device, csa2_ctx** out);
csa2_status csa2_ctx_destroy(csa2_ctx* ctx);
/* Synchronise `stream`, then return (and clear) the status kernels recorded:
   CSA2_OK, CSA2_ERR_DEVICE or CSA2_ERR_TIMEOUT; CSA2_ERR_CUDA if the stream
   itself reports an error. */
csa2_status csa2_ctx_check(csa2_ctx* ctx, void* stream);

/* Failure-detection test hook.  The next tensor-core launch on this context (an
   indexer scan, or the sparse attention's tensor-core kernel) runs with a producer
   that never signals its consumers (the scan's key copies, the attention's query
   images), whose bounded waits then expire after `budget_cycles` (0 = the default
   of 2^31 cycles) and record CSA2_ERR_TIMEOUT; the kernel waits for the copies it
   did issue, frees its tensor memory and exits, and the context stays usable.  The
   flag clears after that one launch.  The selection kernels have no waits to
   expire: their only synchronisation is the hardware barrier of a co-scheduled
   thread-block cluster. */
csa2_status csa2_ctx_test_stall_next(csa2_ctx* ctx, long long budget_cycles);

/*
 * csa2_compress -- gated token compressor with its write epilogue.
 *
 * Non-overlapping form (cb == NULL): Attention-evolution page §4.1 and
 * DSA-to-CSA/HCA page eqs. (22)-(23):
 *     E[i, ch] = sum_{j<m} softmax_j(za[m i + j, ch] + ba[j, ch]) * ca[m i + j, ch]
 * Overlapping form (cb != NULL): DSA-to-CSA/HCA page eqs. (11)-(12): a per-channel
 * softmax over the 2m rows [za[block i] + ba ; zb[block i-1] + bb] weighting
 * [ca[block i] ; cb[block i-1]].  Block 0 has no history (zb = -inf, cb = 0)
 * unless prev_cb/prev_zb carry the previous block's rows (the compressor state
 * of the Attention-evolution page §3.3).
 * Epilogue (Attention-evolution page §4.1): [RMSNorm] -> [RoPE at pos0 + m i]
 * -> store as out_dt (CSA2_FP4_E4M3x16 packs the row).
 *
 * B independent token streams (sequences) are compressed in one call.
 *   ca, za, cb, zb : [B, n_tokens, c] in in_dt (F32 or BF16)
 *   ba, bb         : [m, c] f32, NULL = 0
 *   prev_cb/prev_zb: [B, m, c] in in_dt, or both NULL
 *   pos0           : [B] int64 device array, position of each stream's first token
 *                    (NULL = 0); entry i of stream b sits at pos0[b] + m*i
 *   out            : entry i of stream b goes to row b*out_seq_stride + i of out,
 *                    rows of c values in out_dt (F32, BF16) or c/2 + c/16 bytes
 *                    (CSA2_FP4_E4M3x16) or c/2 + c/32 bytes (CSA2_MXFP4_E8M0x32, the
 *                    indexer-key format); out_seq_stride >= n_tokens/m
 * n_tokens % m == 0, c % 128 == 0, c <= 1024, m >= 1; RoPE acts on the last 64
 * channels.
 */
csa2_status csa2_compress(csa2_ctx* ctx,
                          const void* ca, const void* za, const void* cb, const void* zb,
                          csa2_dtype in_dt, const float* ba, const float* bb,
                          const void* prev_cb, const void* prev_zb,
                          int B, int64_t n_tokens, int c, int m, const int64_t* pos0,
                          float rope_base, unsigned flags, void* out, csa2_dtype out_dt,
                          int64_t out_seq_stride, void* stream);

/*
 * csa2_compress_varlen -- csa2_compress over packed samples (a varlen batch): the
 * tokens of S samples lie back to back, sample s at tokens cu_tokens[s] ..
 * cu_tokens[s+1]-1 of ca/za/cb/zb ([total tokens, c] in in_dt).  Samples never share a
 * compression window (DSA-to-CSA/HCA page, the note under the compressor code and
 * «算法语义»): each is compressed as if alone -- blocks start at its first token, its
 * first block has no history, a tail shorter than m is left out (it is not completed
 * by the next sample).  Entry i of sample s goes to row s*out_seq_stride + i of out at
 * position pos0[s] + m*i (pos0 NULL = 0), so each sample's cache row is its own and the
 * window and the indexer's visible range stay inside the sample.
 *   cu_tokens  : [S+1] int64 device array, non-decreasing, cu_tokens[0] = 0
 *   max_tokens : an upper bound of the tokens of any one sample (sizes the grid)
 *   out_seq_stride >= max_tokens/m when S > 1.  Other arguments as csa2_compress.
 */
csa2_status csa2_compress_varlen(csa2_ctx* ctx,
                                 const void* ca, const void* za, const void* cb, const void* zb,
                                 csa2_dtype in_dt, const float* ba, const float* bb,
                                 int S, const int64_t* cu_tokens, int64_t max_tokens, int c, int m,
                                 const int64_t* pos0, float rope_base, unsigned flags, void* out,
                                 csa2_dtype out_dt, int64_t out_seq_stride, void* stream);

/*
 * csa2_compress_step -- the compressor in decode, one token per sequence per call,
 * with the compressor state of the Attention-evolution page §3.3 (the unfinished
 * block's projections and gate logits; with overlap, the previous block's overlap
 * half).  A compressed entry exists once its block is complete (DSA-to-CSA/HCA page
 * «因果边界与短滑窗»): the token at position p goes to slot p % m of its sequence's
 * state; if p % m == m-1 it completes block i = p/m, and entry i -- the same value
 * csa2_compress computes for the whole sequence, at position m*i -- is written to row
 * b*out_seq_stride + i of out (typically the cache), after which block i's overlap
 * half becomes the history of block i+1.  Positions count from the sequence start.
 *   ca, za, cb, zb : [B, c] this step's rows in in_dt (cb/zb NULL: non-overlap)
 *   ba, bb         : [m, c] f32 or NULL
 *   pos            : [B] int64 device array; pos[b] < 0 skips sequence b this step
 *   state          : caller-owned device memory of csa2_compress_state_bytes()
 *                    bytes (16-byte aligned), per sequence [ca, za (, cb, zb,
 *                    prev cb, prev zb)] x [m, c] in in_dt.  It needs no clearing
 *                    before position 0; csa2_compress_state_seed fills it from a
 *                    prefix of the sequence.
 *   out, out_dt    : as csa2_compress.
 * Calls must be made in position order per sequence; the call only reads and
 * writes device memory on `stream`.
 */
size_t csa2_compress_state_bytes(int B, int c, int m, csa2_dtype in_dt, int overlap);
csa2_status csa2_compress_step(csa2_ctx* ctx,
                               const void* ca, const void* za, const void* cb, const void* zb,
                               csa2_dtype in_dt, const float* ba, const float* bb,
                               int B, int c, int m, const int64_t* pos, void* state,
                               float rope_base, unsigned flags, void* out, csa2_dtype out_dt,
                               int64_t out_seq_stride, void* stream);
/* Seed the state from the first n_tokens tokens of each sequence ([B, n_tokens, c]
 * rows, e.g. a prefill compressed with csa2_compress): the unfinished block's rows
 * and the last complete block's overlap half.  The next step is position n_tokens. */
csa2_status csa2_compress_state_seed(csa2_ctx* ctx,
                                     const void* ca, const void* za, const void* cb, const void* zb,
                                     csa2_dtype in_dt, int B, int64_t n_tokens, int c, int m,
                                     void* state, void* stream);

/*
 * csa2_fp4_pack / csa2_fp4_unpack -- the two 4-bit cache formats.
 *   CSA2_FP4_E4M3x16  (c % 64 == 0): per 16 channels s = E4M3_RNE(amax/6) (satfinite, f32 IEEE
 *                       division); s == 0 -> codes 0; code = E2M1_RNE(x/s), sat. +-6.
 *   CSA2_MXFP4_E8M0x32 (c % 128 == 0): per 32 values X = 2^(floor(log2 amax) - 2) as E8M0,
 *                       amax == 0 -> scale byte 0, codes 0; code = E2M1_RNE(x/X).
 * x: [rows, c] in x_dt (F32 or BF16); packed row r is written at out + r*out_ld
 * (out_ld in bytes, a multiple of 4, >= the row size; 0 = rows back to back), so a
 * batch of new rows can go straight into per-sequence cache slots.  Unpack reads
 * back-to-back rows and writes F32 or BF16 (exact: every FP4 value times its scale
 * fits in bf16).
 */
csa2_status csa2_fp4_pack(csa2_ctx* ctx, const void* x, csa2_dtype x_dt, int64_t rows, int c,
                          csa2_dtype fmt, uint8_t* out, int64_t out_ld, void* stream);
csa2_status csa2_fp4_unpack(csa2_ctx* ctx, const uint8_t* in, csa2_dtype fmt, int64_t rows,
                            int c, void* out, csa2_dtype out_dt, void* stream);

/*
 * csa2_visible_entries -- the causal rule of the compressed cache (DSA-to-CSA/HCA
 * page, «因果边界与短滑窗»): compressed entry j (made from tokens mj .. mj+m-1) is
 * visible to the query at position t iff t >= m(j+1), so a query sees
 *     n_visible[i] = floor(q_pos[i] / m)      (0 for a negative position)
 * entries.  The n_visible arrays the indexer, the selections and the dense attention
 * take are this.
 *   q_pos     : [rows] int64, device
 *   n_visible : [rows] int64, device (may alias q_pos)
 *   m >= 1.  Asynchronous on `stream`; invalid arguments return before any launch.
 */
csa2_status csa2_visible_entries(csa2_ctx* ctx, const int64_t* q_pos, int64_t rows, int m, int64_t* n_visible,
                                 void* stream);

/*
 * csa2_index_score -- Lightning-indexer scores (DSA-to-CSA/HCA page eq. (16)):
 *     I[b,q,s] = sum_h w[b,q,h] * ReLU(q_idx[b,q,h,:] . k_idx[b,s,:])
 * with no scale and no softmax, for the entries visible to the query
 * (s < n_visible[b,q]; the causal rule t >= m(j+1) gives n_visible = floor(t/m)).
 *
 *   q_idx  : [B, Q, H_I, d_I] in q_dt (F32 or BF16), or [B, Q, H_I, 68] B with
 *            q_dt = CSA2_MXFP4_E8M0x32 (packed by csa2_fp4_pack like the keys)
 *   w      : [B, Q, H_I] f32
 *   k_idx  : [B, N, d_I] in k_dt (F32, BF16) or [B, N, d_I/2 + d_I/32] B (MXFP4)
 *   n_visible : [B, Q] int64, device
 * Full scan (pool_blocks == NULL):
 *   scores    : [B, Q, N] f32 or NULL; entries s >= n_visible get -inf
 *   block_max : [B, Q, ceil(N/block)] f32 or NULL: max over the visible members of
 *               each block of `block` entries (CSA2 page, «解码器里的分层索引»);
 *               blocks with no visible member get -inf
 *   block_hist: [B, Q, CSA2_BLOCK_HIST_BINS] uint32 or NULL (needs block_max): a
 *               summary of each row's visible block maxima that csa2_block_pool
 *               takes to pick its pool with fewer passes (opaque: counts of the
 *               maxima by their leading bits).  Written in full by this call.
 * Candidate mode (Reindex, CSA2 page «三种模式» and «解码器里的分层索引»):
 *   pool_blocks : [B, Q, n_pool] int32 block ids (-1 = empty slot)
 *   scores      : [B, Q, n_pool*block] f32 (required); candidate c is entry
 *                 pool[c/block]*block + c%block; invalid candidates get -inf
 *   block_max must be NULL.
 * d_I == 128, 1 <= H_I <= 128, block a power of two <= 32, B*Q <= 65535.
 *
 * Paths.  MXFP4 queries over MXFP4 keys with H_I == 64, block == 8, N % 8 == 0 (and
 * n_pool % 16 == 0) run the QK product in FP4 on the tensor cores (the page puts the
 * indexer QK path in FP4, «Lightning Indexer：公式 (13)–(17)»): E2M1 products with
 * their E8M0 block scales, fp32 accumulation.  BF16 queries over BF16 or MXFP4 keys
 * on the same shapes use the bf16/f16 tensor-core scan (exact products, fp32 sums).
 * Everything else runs on the CUDA cores in fp32.
 */
#define CSA2_BLOCK_HIST_BINS 4096
csa2_status csa2_index_score(csa2_ctx* ctx,
                             const void* q_idx, csa2_dtype q_dt, const float* w,
                             const void* k_idx, csa2_dtype k_dt,
                             int B, int Q, int64_t N, int H_I, int d_I,
                             const int64_t* n_visible,
                             const int32_t* pool_blocks, int n_pool, int block,
                             float* scores, float* block_max, uint32_t* block_hist, void* stream);

/*
 * csa2_index_score_mxq -- the full scan of csa2_index_score on its FP4 QK path
 * (DSA-to-CSA/HCA page, «Lightning Indexer：公式 (13)–(17)»: the indexer QK product in
 * FP4) from a bf16 indexer query: each query head row is packed to MXFP4 inside the
 * scan by the rule of csa2_fp4_pack (so no separate packing launch), then scored as
 * csa2_index_score scores a packed query, with the same outputs.
 *   q_bf16   : [B, Q, 64, 128] bf16 (16-byte aligned)
 *   k_idx    : [B, N, 68] B MXFP4 indexer keys; N a multiple of 8; block == 8
 *   q_mx_out : [B, Q, 64, 68] B or NULL: the packed query bytes, as csa2_fp4_pack
 *              writes them (4-byte aligned)
 * w, n_visible, scores, block_max, block_hist: as csa2_index_score's full scan.
 * Other head counts, head sizes or blocks return CSA2_ERR_UNSUPPORTED (pack the query
 * with csa2_fp4_pack and call csa2_index_score).
 */
csa2_status csa2_index_score_mxq(csa2_ctx* ctx, const void* q_bf16, const float* w, const void* k_idx,
                                 int B, int Q, int64_t N, int H_I, int d_I, const int64_t* n_visible,
                                 int block, float* scores, float* block_max, uint32_t* block_hist,
                                 uint8_t* q_mx_out, void* stream);

/*
 * csa2_topk -- top-k selection/*
 * csa2_topk -- top-k selection (DSA-to-CSA/HCA page eq. (17)) in one total order:
 * score descending, entry index ascending (the lower index wins a tie).
 * Row r of `scores` (stride ld floats) covers:
 *   full mode (pool_blocks == NULL): entries 0 .. n_visible[r]-1;
 *   candidate mode: candidate c -> entry pool_blocks[r, c/block]*block + c%block,
 *                   valid if that block id >= 0 and the entry < n_visible[r].
 * If a row has <= k valid elements, all are returned.  -0.0 equals +0.0.
 *   out_idx   : [rows, k] int32 entry ids, ascending, padded with -1
 *   out_score : [rows, k] f32 matching scores (-inf in padding), or NULL
 * Scores must be finite (NaN order is unspecified).  1 <= k <= 4096.
 */
csa2_status csa2_topk(csa2_ctx* ctx, const float* scores, int64_t rows, int64_t n, int64_t ld,
                      const int64_t* n_visible, const int32_t* pool_blocks, int n_pool,
                      int block, int k, int32_t* out_idx, float* out_score,
                      void* ws, size_t ws_bytes, void* stream);
/* Workspace of the selections (csa2_topk, csa2_block_pool): when rows are few and
   long, each row is split over several CTAs that keep their chunk's top-k in `ws`
   (caller-owned device memory, 16-byte aligned) for an exact merge.  The
   *_workspace_bytes functions give the size that enables it; with a smaller or NULL
   workspace a row is handled by one CTA (same result, slower).  rows <= 65535. */
size_t csa2_topk_workspace_bytes(csa2_ctx* ctx, int64_t rows, int64_t n, int k);

/*
 * csa2_block_pool -- candidate pool of the hierarchical sparse indexer (CSA2 page,
 * «解码器里的分层索引»; Attention-evolution page §4.4): blocks of `block` entries,
 * block score = the block max (from csa2_index_score); the newest visible block
 * floor((V-1)/block) is always kept and the remaining n_keep-1 slots go to the best
 * other blocks by (block max desc, block id asc).  If ceil(V/block) <= n_keep,
 * every visible block is kept; V == 0 gives an all -1 row.
 *   block_max  : [rows, ld] f32 (first ceil(V/block) used)
 *   block_hist : [rows, CSA2_BLOCK_HIST_BINS] from csa2_index_score over the same
 *                block maxima, or NULL (then the call builds it in `ws`, if it fits)
 *   n_visible  : [rows] int64 (V per row)
 *   out_blocks : [rows, n_keep] int32 ascending, -1 padded.   1 <= n_keep <= 4096.
 *   out_top    : [rows, n_top] int32 or NULL: the n_top best visible blocks by
 *                (block max desc, block asc) -- no block is forced in -- ascending,
 *                -1 padded.  The top-k entries of the row (k <= n_top) all lie in these
 *                blocks: every block ranked above a block b holds an entry, its
 *                maximum, that ranks above every entry of b.  So csa2_topk over the
 *                candidates of out_top gives the row's top-k.  Needs a histogram
 *                (block_hist or a workspace that holds one); n_top <= n_keep - 1.
 * With a histogram the selection reads the maxima once and resolves the threshold
 * from the histogram; without one it runs the general radix select.
 */
csa2_status csa2_block_pool(csa2_ctx* ctx, const float* block_max, const uint32_t* block_hist,
                            int64_t rows, int64_t ld, const int64_t* n_visible, int block, int n_keep,
                            int32_t* out_blocks, int32_t* out_top, int n_top,
                            void* ws, size_t ws_bytes, void* stream);
size_t csa2_block_pool_workspace_bytes(csa2_ctx* ctx, int64_t rows, int64_t ld, int n_keep);

/* The histogram csa2_index_score writes beside the block maxima, built from block
   maxima that came from elsewhere ([rows, ld] f32, n_visible entries per row):
   block_hist [rows, CSA2_BLOCK_HIST_BINS] uint32 (16-byte aligned), written in full. */
csa2_status csa2_block_hist(csa2_ctx* ctx, const float* block_max, int64_t rows, int64_t ld,
                            const int64_t* n_visible, int block, uint32_t* block_hist, void* stream);

/*
 * csa2_pool_topk -- the selections of a Full decode layer in one call: the block pool
 * of csa2_block_pool (for the Reindex layers that follow) and the layer's own top-k
 * entries (DSA-to-CSA/HCA page eq. (17); CSA2 page, «解码器里的分层索引»), from the
 * scan's block maxima, their histogram and the stored entry scores.  The top-k entries
 * lie in the k best blocks (every block ranked above a block b holds an entry, its
 * maximum, that ranks above every entry of b), and each of them scores at least the
 * smallest of those k maxima, so only those blocks' entries above that value are
 * ranked; the result equals csa2_topk over all the row's scores.
 *   block_max, block_hist : as csa2_block_pool (block_hist from csa2_index_score)
 *   scores     : [rows, n_ent] f32, the full-scan scores (entries < n_visible read)
 *   out_blocks : [rows, n_keep] int32 (the pool);  out_idx : [rows, k] int32 entry
 *                ids ascending, -1 padded;  out_score : [rows, k] f32 or NULL
 * 2 <= n_keep <= 4096, 1 <= k <= n_keep - 1, k * block <= 8192, block <= 16,
 * ld <= 262,144.  Other shapes return CSA2_ERR_UNSUPPORTED (csa2_block_pool and
 * csa2_topk serve them).
 */
csa2_status csa2_pool_topk(csa2_ctx* ctx, const float* block_max, const uint32_t* block_hist,
                           const float* scores, int64_t rows, int64_t ld, int64_t n_ent,
                           const int64_t* n_visible, int block, int n_keep, int k,
                           int32_t* out_blocks, int32_t* out_idx, float* out_score, void* stream);

/*
 * csa2_sparse_attn -- shared-KV MQA over the selected compressed entries plus the
 * sliding window (DSA-to-CSA/HCA page eqs. (18)-(19), (27), «因果边界与短滑窗»;
 * CSA2 page «保留了 CSA 的骨架»).  For query (b,q) at position t = q_pos[b,q] and
 * head i, the key/value rows are
 *     { kv[b, s] : s in idx[b,q,:], s != -1 }  U  { window rows at positions
 *       max(0, t-window+1) .. t, slot (p - swa_pos0) mod swa_cap of swa[b] }.
 * With the default flags: q^ = RoPE_t(RMSNorm(q)), k^_j = RMSNorm(row_j) (stored
 * rows are already rotated at their own positions), z_j = q^.k^_j / sqrt(c),
 * p_j = e^{z_j} / (sum_l e^{z_l} + e^{sink_i}),  out = RoPE_{-t}(sum_j p_j k^_j).
 * Reuse layers call this with an upstream layer's idx (no indexer).
 *
 *   q     : [B, Q, H, c] in q_dt (F32 or BF16)
 *   kv    : [B, N, c] (F32, BF16) or [B, N, c/2 + c/16] B (CSA2_FP4_E4M3x16)
 *   idx   : [B, Q, k] int32, -1 = none; ids outside [0, N) are skipped and flagged
 *   swa   : [B, swa_cap, c] in swa_dt (F32 or BF16); window <= swa_cap
 *   q_pos : [B, Q] int64
 *   sink  : [H] f32 or NULL (no sink term)
 *   out   : [B, Q, H, c] in out_dt (F32 or BF16);  lse: [B, Q, H] f32 or NULL,
 *           lse = log(sum_j e^{z_j} + e^{sink_i})
 * c == 512, 1 <= H <= 128, 0 <= k <= 2048, 0 <= window <= 1024, B*Q <= 65535.
 *
 * Two paths compute this.  The tensor-core path (tcgen05) runs when q and swa are
 * BF16, kv is BF16 or FP4, both RMSNorm flags are set, H <= 64 and the workspace
 * holds at least csa2_sparse_attn_workspace_bytes(); it rounds the normalised,
 * rotated query and the probabilities to bf16 for the MMAs (fp32 accumulation) and,
 * because both norms bound every logit by sqrt(c), uses the fixed softmax offset 24
 * instead of a running maximum.  Every other call takes the CUDA-core path, which
 * works in fp32 throughout.
 *
 * Workspace (caller-owned device memory, 16-byte aligned): the tensor-core path keeps
 * each query's prepared bf16 image there (64 KB per query), with few queries the
 * per-split partial results of its key split, and, when the call gathers each row
 * many times over (B*Q*(k+window) >= 4*(B*N + B*swa_cap), as in prefill), the rows'
 * RMS factors computed once per call; the CUDA-core path keeps only its key-split
 * partials.  csa2_sparse_attn_workspace_bytes(), given the same N and swa_cap as the
 * call, returns the size that enables all of it; the tensor-core path runs without
 * the factor table when only it is missing, and with less than the images and
 * partials the call falls back to the CUDA-core path with as many splits as fit
 * (NULL: no split).  Calls that share a workspace must not overlap on the GPU.
 */
size_t csa2_sparse_attn_workspace_bytes(csa2_ctx* ctx, int B, int Q, int H, int k, int window, int64_t N,
                                        int64_t swa_cap);
csa2_status csa2_sparse_attn(csa2_ctx* ctx,
                             const void* q, csa2_dtype q_dt,
                             const void* kv, csa2_dtype kv_dt, int64_t N,
                             const int32_t* idx, int k,
                             const void* swa, csa2_dtype swa_dt, int64_t swa_cap,
                             int64_t swa_pos0, int window,
                             const int64_t* q_pos, const float* sink,
                             int B, int Q, int H, int c, float rope_base, unsigned flags,
                             void* out, csa2_dtype out_dt, float* lse,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_attn_prepare -- the query half of csa2_sparse_attn / csa2_dense_attn ahead of
 * time: each query head RMS-normalised and rotated by RoPE_t (the q^ of the
 * attention), as the tensor-core path's bf16 operand image, and the RoPE table of
 * the query positions, into `ws`.  It depends only on q and q_pos, so it can run
 * beside the indexer and the selection (another stream) instead of after them.  The
 * attention call then passes the same sizes, flags | CSA2_ATTN_PREPARED and the same
 * workspace, which must not be touched in between.  Sizes and flags as the attention
 * call (its k, window, N and swa_cap place the image in the workspace); H <= 64.
 * When that call does not take the tensor-core path it ignores the prepared image.
 */
csa2_status csa2_attn_prepare(csa2_ctx* ctx, const void* q, csa2_dtype q_dt, const int64_t* q_pos,
                              int B, int Q, int H, int c, int k, int window, int64_t N, int64_t swa_cap,
                              float rope_base, unsigned flags, void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_dense_attn -- the HCA attention (DSA-to-CSA/HCA page «HCA：公式 (20)–(26)»,
 * eq. (26); window of «因果边界与短滑窗»): with the heavily compressed cache (m' = 128,
 * produced by csa2_compress), each query attends densely over every visible
 * compressed entry instead of an indexer's selection.  The computation is exactly
 * csa2_sparse_attn with idx = 0 .. n_visible[b,q]-1, plus the same window, sink,
 * norms and rotations.
 *   n_visible : [B, Q] int64, entries 0 .. n_visible-1 of sequence b are taken (the
 *               causal rule gives n_visible = floor(t/m'))
 *   k_max     : an upper bound of n_visible (at most 4,194,304); it sizes the key
 *               splits, so csa2_sparse_attn_workspace_bytes(ctx, B, Q, H, k_max, window,
 *               N, swa_cap) gives the workspace
 * Every other argument, layout and error as csa2_sparse_attn.
 */
csa2_status csa2_dense_attn(csa2_ctx* ctx,
                            const void* q, csa2_dtype q_dt,
                            const void* kv, csa2_dtype kv_dt, int64_t N,
                            const int64_t* n_visible, int k_max,
                            const void* swa, csa2_dtype swa_dt, int64_t swa_cap, int64_t swa_pos0,
                            int window, const int64_t* q_pos, const float* sink,
                            int B, int Q, int H, int c, float rope_base, unsigned flags,
                            void* out, csa2_dtype out_dt, float* lse,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_sparse_attn_noalloc -- csa2_sparse_attn for callers that may not allocate
 * device memory.  The paper has no counterpart: this is a deployment convenience.
 *
 * Hosts that manage all device memory themselves (a serving engine that reserves
 * one arena at start-up and does not let plugins call cudaMalloc, or a loop that
 * cannot afford an allocation's latency and implicit synchronisation) cannot pass
 * the split-key workspace.  This entry point takes the same arguments minus the
 * workspace and keeps the partial results in a device array compiled into the
 * library, CSA2_NOALLOC_SCRATCH_BYTES large; every GPU that loads the library holds
 * that array until the process exits.  It calls no allocator.
 *   - The first call with a context looks up the array's device address on the
 *     context's device (a one-time set-up that allocates nothing) and keeps it in
 *     the context; make that first call before any stream capture.  After a device
 *     reset the context must be created again (the array may have moved).
 *   - All calls share the array: calls whose kernels overlap on the GPU race.
 *     Nothing in it needs to start at zero (each call rewrites what it reads).
 *   - The tensor-core path is taken when its workspace fits the array, so results
 *     equal csa2_sparse_attn's with a full workspace whenever that workspace is at
 *     most CSA2_NOALLOC_SCRATCH_BYTES.  Otherwise the CUDA-core path runs with its
 *     key split in the array; that split needs fewer than
 *     2 * (4 * SMs) * 8 * 516 * 4 bytes (20,078,592 on a 152-SM part), so it always
 *     fits there.  On a part with more SMs, a call whose split would need more than
 *     CSA2_NOALLOC_SCRATCH_BYTES is rejected with CSA2_ERR_INVALID_ARG before
 *     anything is launched.
 */
#define CSA2_NOALLOC_SCRATCH_BYTES (24u << 20)
csa2_status csa2_sparse_attn_noalloc(csa2_ctx* ctx,
                                     const void* q, csa2_dtype q_dt,
                                     const void* kv, csa2_dtype kv_dt, int64_t N,
                                     const int32_t* idx, int k,
                                     const void* swa, csa2_dtype swa_dt, int64_t swa_cap,
                                     int64_t swa_pos0, int window,
                                     const int64_t* q_pos, const float* sink,
                                     int B, int Q, int H, int c, float rope_base, unsigned flags,
                                     void* out, csa2_dtype out_dt, float* lse, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
