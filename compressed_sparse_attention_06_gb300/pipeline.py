"""Per-layer steps of the CSA2 hot path, strung from the C-ABI entry points.

Every arithmetic step runs in libcsa2.so; this module only allocates outputs
(torch device memory) and orders the calls on the current stream.

Layer modes (CSA2 page, «三种模式：谁算、谁复用»):
  Full    -- own indexer over all visible entries (+ block pool in the decoder),
  Reindex -- own indexer over the pooled candidates only,
  Reuse   -- upstream indices, attention only.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import csa2 as C

TOPK = 512
POOL_BLOCK = 8
POOL_KEEP = 2048


def visible_entries(q_pos: torch.Tensor, m: int) -> torch.Tensor:
    """Entries visible to each query: entry j needs t >= m(j+1), so floor(t/m)
    (DSA-to-CSA/HCA page, «因果边界与短滑窗»); computed by csa2_visible_entries."""
    return C.csa2_visible_entries(q_pos, m)


@dataclass
class DecodeBuffers:
    """Preallocated outputs of a Full-mode decode step (reused across steps)."""
    scores: torch.Tensor         # the full scan's scores (the top-k reads its best blocks' entries)
    block_max: torch.Tensor
    block_hist: torch.Tensor     # the scan's summary of the block maxima, for the pool
    pool: torch.Tensor
    top_blocks: torch.Tensor     # the best top_n blocks: the top-k entries lie in them
    cand_scores: torch.Tensor
    idx: torch.Tensor
    out: torch.Tensor
    attn_ws: torch.Tensor
    pool_ws: torch.Tensor
    topk_ws: torch.Tensor
    qI_mx: torch.Tensor          # the indexer query packed to MXFP4 (FP4 QK path)


def top_blocks_for(k: int) -> int:
    """Blocks the top-k selection rescores: the k best blocks hold the top-k entries
    (every block ranked above a block b holds its maximum, which ranks above every
    entry of b), rounded up to a whole candidate tile of 32 blocks."""
    return (k + 31) // 32 * 32


def alloc_decode(B: int, Q: int, N: int, H: int, c: int, device, out_dtype=torch.bfloat16,
                 k: int = TOPK, block: int = POOL_BLOCK, n_keep: int = POOL_KEEP,
                 window: int = 128, h_idx: int = 64) -> DecodeBuffers:
    nb = (N + block - 1) // block
    n_top = top_blocks_for(k)
    return DecodeBuffers(
        scores=C.alloc((B, Q, N), dtype=torch.float32, device=device),
        block_max=C.alloc((B, Q, nb), dtype=torch.float32, device=device),
        block_hist=C.alloc((B, Q, C.BLOCK_HIST_BINS), dtype=torch.int32, device=device),
        pool=C.alloc((B, Q, n_keep), dtype=torch.int32, device=device),
        top_blocks=C.alloc((B, Q, n_top), dtype=torch.int32, device=device),
        cand_scores=C.alloc((B, Q, n_top * block), dtype=torch.float32, device=device),
        idx=C.alloc((B, Q, k), dtype=torch.int32, device=device),
        out=C.alloc((B, Q, H, c), dtype=out_dtype, device=device),
        attn_ws=C.alloc(max(16, C.csa2_sparse_attn_workspace_bytes(B, Q, H, k, window,
                                                                       torch.device(device).index, N=N,
                                                                       swa_cap=window)),
                            dtype=torch.uint8, device=device),
        pool_ws=C._ws(C.csa2_block_pool_workspace_bytes(B * Q, nb, n_keep, torch.device(device).index), device),
        topk_ws=C._ws(C.csa2_topk_workspace_bytes(B * Q, n_top * block, k, torch.device(device).index), device),
        qI_mx=C.alloc((B, Q, h_idx, C.mxfp4_row_bytes(128)), dtype=torch.uint8, device=device),
    )


def full_decode_step(qI, w, kI, q, kv, swa, q_pos, n_visible, sink, buf: DecodeBuffers, *,
                     window: int = 128, swa_pos0: int = 0, k: int = TOPK, block: int = POOL_BLOCK,
                     n_keep: int = POOL_KEEP, flags: int = C.ATTN_DEFAULT,
                     side_stream: Optional[torch.cuda.Stream] = None):
    """Full layer with the hierarchical pool (CSA2 page, «解码器里的分层索引»):
    scan all visible entries (scores, block maxima and their histogram), pick the
    pool (for the Reindex layers that follow) and the layer's own top-k in one call
    (the top-k of all entries lies inside the k best blocks, which lie inside the
    pool), and attend over the selected entries plus the window.  Shapes that call
    does not take run the pool, the best blocks' rescoring and the top-k one by one.

    With an MXFP4 indexer cache the QK product runs in FP4 (DSA-to-CSA/HCA page,
    «Lightning Indexer：公式 (13)–(17)»): a bf16/f32 qI is first packed to MXFP4 by
    the same rule as the keys (into buf.qI_mx); an already packed uint8 qI is used
    as given.

    side_stream: the attention's query half (csa2_attn_prepare) runs there, beside
    the selection, after the scan (which fills the GPU by itself)."""
    fused = pool_topk_applies(k, block, n_keep, buf.block_max.shape[-1])
    if mxq_applies(qI, kI, block):
        # the FP4 QK path with the query packed inside the scan (packed bytes kept in buf)
        C.csa2_index_score_mxq(qI, w, kI, n_visible, block=block, scores=buf.scores if fused else None,
                               want_scores=fused, want_block_max=True, block_max=buf.block_max,
                               block_hist=buf.block_hist, q_mx_out=buf.qI_mx)
        qI = buf.qI_mx
    else:
        qI = mxfp4_query(qI, kI, buf.qI_mx)
        C.csa2_index_score(qI, w, kI, n_visible, block=block, scores=buf.scores if fused else None,
                           want_scores=fused, want_block_max=True, block_max=buf.block_max,
                           block_hist=buf.block_hist)
    B, Q, H = q.shape[:3]
    prepared = side_stream is not None and H <= 64
    if prepared:
        side_stream.wait_stream(torch.cuda.current_stream(q.device))
        with torch.cuda.stream(side_stream):
            C.csa2_attn_prepare(q, q_pos, buf.attn_ws, k, window=window, N=kv.shape[1], swa_cap=swa.shape[1],
                                flags=flags)
    if fused:
        C.csa2_pool_topk(buf.block_max, buf.block_hist, buf.scores, n_visible, k, block=block, n_keep=n_keep,
                         out=buf.pool, out_idx=buf.idx)
    else:
        C.csa2_block_pool(buf.block_max, n_visible, block=block, n_keep=n_keep, out=buf.pool, ws=buf.pool_ws,
                          block_hist=buf.block_hist, n_top=buf.top_blocks.shape[-1], out_top=buf.top_blocks)
        C.csa2_index_score(qI, w, kI, n_visible, pool=buf.top_blocks, block=block, scores=buf.cand_scores)
        C.csa2_topk(buf.cand_scores, n_visible, k, pool=buf.top_blocks, block=block, out_idx=buf.idx,
                    ws=buf.topk_ws)
    if prepared:
        torch.cuda.current_stream(q.device).wait_stream(side_stream)
    C.csa2_sparse_attn(q, kv, buf.idx, swa, q_pos, sink, window=window, swa_pos0=swa_pos0,
                       flags=flags | (C.ATTN_PREPARED if prepared else 0), out=buf.out, ws=buf.attn_ws)
    return buf


def pool_topk_applies(k: int, block: int, n_keep: int, n_blocks: int) -> bool:
    """The shapes csa2_pool_topk takes (its header states them)."""
    chunk = -(-(-(-n_blocks // 16)) // 1024) * 1024
    return 1 <= k <= n_keep - 1 and k * block <= 8192 and block <= 16 and chunk <= 16384


def mxq_applies(qI, kI, block: int) -> bool:
    """Shapes csa2_index_score_mxq takes: a bf16 query of 64 heads x 128 over MXFP4 keys,
    blocks of 8, a cache length that is a multiple of 8."""
    return (qI.dtype == torch.bfloat16 and kI.dtype == torch.uint8 and tuple(qI.shape[2:]) == (64, 128)
            and block == 8 and kI.shape[1] % 8 == 0)


def mxfp4_query(qI, kI, out=None):
    """The indexer query as the scan takes it: packed to MXFP4 when the keys are
    MXFP4 (uint8 rows) and the query is not packed yet; unchanged otherwise."""
    if kI.dtype != torch.uint8 or qI.dtype == torch.uint8:
        return qI
    return C.csa2_fp4_pack(qI, C.MXFP4_E8M0x32, out=out)


def reindex_step(qI, w, kI, pool, n_visible, cand_scores=None, idx=None, k: int = TOPK, block: int = POOL_BLOCK):
    """Reindex layer: own indexer query over the pooled candidates, then top-k
    (FP4 QK product over an MXFP4 cache, as in full_decode_step)."""
    qI = mxfp4_query(qI, kI)
    sc, _ = C.csa2_index_score(qI, w, kI, n_visible, pool=pool, block=block, scores=cand_scores)
    ids, _ = C.csa2_topk(sc, n_visible, k, pool=pool, block=block, out_idx=idx)
    return ids


def reuse_attention(q, kv, idx, swa, q_pos, sink, out=None, window: int = 128, swa_pos0: int = 0,
                    flags: int = C.ATTN_DEFAULT):
    """Reuse layer (and the attention of Full/Reindex layers): upstream indices, own
    query and own window."""
    o, _ = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, swa_pos0=swa_pos0, flags=flags,
                              out=out)
    return o


def full_topk_step(qI, w, kI, n_visible, k: int = TOPK, scores=None, idx=None):
    """Full layer without a pool (encoder / prefill): full scores, then top-k
    (FP4 QK product over an MXFP4 cache, as in full_decode_step)."""
    qI = mxfp4_query(qI, kI)
    sc, _ = C.csa2_index_score(qI, w, kI, n_visible, scores=scores)
    ids, _ = C.csa2_topk(sc, n_visible, k, out_idx=idx)
    return sc, ids


@dataclass
class PrefillBuffers:
    scores: torch.Tensor
    idx: torch.Tensor
    out: torch.Tensor
    n_visible: torch.Tensor
    attn_ws: torch.Tensor
    topk_ws: torch.Tensor


def alloc_prefill(Q: int, N: int, H: int, c: int, device, q_pos: torch.Tensor, m: int,
                  out_dtype=torch.bfloat16, k: int = TOPK, window: int = 128, swa_cap: int = 0) -> PrefillBuffers:
    """swa_cap: rows of the window buffer the attention will read (sizes the workspace
    for the per-call table of row RMS factors)."""
    return PrefillBuffers(
        scores=C.alloc((1, Q, N), dtype=torch.float32, device=device),
        idx=C.alloc((1, Q, k), dtype=torch.int32, device=device),
        out=C.alloc((1, Q, H, c), dtype=out_dtype, device=device),
        n_visible=visible_entries(q_pos, m),
        attn_ws=C.alloc(max(16, C.csa2_sparse_attn_workspace_bytes(1, Q, H, k, window,
                                                                       torch.device(device).index, N=N,
                                                                       swa_cap=swa_cap)),
                            dtype=torch.uint8, device=device),
        topk_ws=C._ws(C.csa2_topk_workspace_bytes(Q, N, k, torch.device(device).index), device),
    )


def prefill_chunk_step(Ca, Cb, Za, Zb, Ba, Bb, prev_Cb, prev_Zb, kv_cache, n_ctx_entries: int, pos0: torch.Tensor,
                       m: int, qI, w, kI, q, swa, swa_pos0: int, q_pos, sink, buf: PrefillBuffers, *,
                       k: int = TOPK, window: int = 128, write_flags: int = C.W_NORM | C.W_ROPE):
    """Encoder prefill chunk (Full layer): the overlapped compressor turns the chunk's
    tokens into new cache entries (carrying the previous block's state), then every
    query of the chunk scores all entries it can see, takes its top-k and attends
    over them plus its window."""
    C.csa2_compress(Ca, Za, m, cb=Cb, zb=Zb, ba=Ba, bb=Bb, prev_cb=prev_Cb, prev_zb=prev_Zb, pos0=pos0,
                    flags=write_flags, out=kv_cache[0, n_ctx_entries:], out_seq_stride=0)
    qI = mxfp4_query(qI, kI)
    C.csa2_index_score(qI, w, kI, buf.n_visible, scores=buf.scores)
    C.csa2_topk(buf.scores, buf.n_visible, k, out_idx=buf.idx, ws=buf.topk_ws)
    C.csa2_sparse_attn(q, kv_cache, buf.idx, swa, q_pos, sink, window=window, swa_pos0=swa_pos0, out=buf.out,
                       ws=buf.attn_ws)
    return buf
