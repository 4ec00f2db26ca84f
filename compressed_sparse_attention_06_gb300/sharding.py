"""Host-side logic for running the path on several GPUs (one process per GPU).

Two ways to split the work, neither needing a data-path collective for the first:

* by sequence (what bench.py does under torchrun): rank r owns sequences
  [r*B, (r+1)*B); every rank runs the whole step on its own sequences and the
  job's time is the maximum over ranks (weak scaling);
* by entry range, for one very long sequence: rank r holds and scans entries
  [lo_r, hi_r) (edges on block boundaries, so no pool block straddles two ranks),
  keeps its own block pool (block ids + block maxima) and its own top-k (global
  ids + scores), and attends over its share of the selected rows without the
  sink, returning (o_r, lse_r).  One all-gather of the small per-rank results
  (n_keep block keys and k entry keys per query) then gives the exact answer:
  the pool and the top-k of the union of the per-rank lists in the same total
  orders, and the log-sum-exp combination of the partial attention outputs with
  the sink added once.

Why the merges are exact (CSA2 page, «解码器里的分层索引», for the pool and its
newest block): a block among the n_keep-1 best of all blocks other than the
newest has fewer than n_keep-1 such blocks ranked above it, so it is also among
the best n_keep-1 of its own rank's blocks, which that rank's pool holds (a
rank's pool forces in its own last block, and best-(n_keep-1)-of-the-rest plus
that block contains the best n_keep-1 of all its blocks).  Likewise an entry of
the global top-k is in its rank's top-k, and a rank's top-k lies inside its
pool, because every block ranked above a block b contributes its maximum entry,
which ranks above every entry of b.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import torch

from . import csa2 as C


def sequences_for_rank(rank: int, world: int, per_rank: int) -> Tuple[int, int]:
    """(first global sequence index, count) owned by `rank`."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return rank * per_rank, per_rank


def entry_range(rank: int, world: int, n_entries: int, align: int = 1) -> Tuple[int, int]:
    """Contiguous entry range [lo, hi) of `rank`, split as evenly as possible in
    units of `align` entries (align = the pool's block size keeps every block on
    one rank); the last range ends at n_entries."""
    if not 0 <= rank < world or align < 1:
        raise ValueError("rank out of range or align < 1")
    units = (n_entries + align - 1) // align
    base, extra = divmod(units, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return min(lo * align, n_entries), min(hi * align, n_entries)


def max_over_ranks(value: float, device: Optional[torch.device] = None) -> float:
    """Maximum of a per-rank number over the process group (identity without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def merge_topk(ids: Sequence[torch.Tensor], scores: Sequence[torch.Tensor], k: int) -> torch.Tensor:
    """Exact merge of per-rank top-k lists (global entry ids, -1 padded, with their
    scores): the k best of the union by (score desc, id asc), ascending, -1 padded."""
    i = torch.cat([t.reshape(-1).to(torch.int64) for t in ids])
    s = torch.cat([t.reshape(-1).to(torch.float64) for t in scores])
    keep = i >= 0
    i, s = i[keep], s[keep]
    order = torch.sort(i, stable=True).indices              # id ascending ...
    i, s = i[order], s[order]
    order = torch.sort(-s, stable=True).indices             # ... then score descending
    best = torch.sort(i[order][:k]).values
    out = torch.full((k,), -1, dtype=torch.int64)
    out[: best.numel()] = best
    return out


def merge_pool(block_ids: Sequence[torch.Tensor], block_max: Sequence[torch.Tensor], n_visible: int,
               block: int = 8, n_keep: int = 2048) -> torch.Tensor:
    """Exact merge of per-rank block pools (global block ids, -1 padded, with their
    block maxima) into the pool of the whole sequence: the newest visible block
    floor((V-1)/block) is always kept, the other n_keep-1 slots go to the best
    gathered blocks by (block max desc, block id asc); if every visible block fits
    (ceil(V/block) <= n_keep) all are kept.  Ascending, -1 padded."""
    V = int(n_visible)
    out = torch.full((n_keep,), -1, dtype=torch.int64)
    if V <= 0:
        return out
    nb = (V + block - 1) // block
    if nb <= n_keep:
        out[:nb] = torch.arange(nb)
        return out
    i = torch.cat([t.reshape(-1).to(torch.int64).cpu() for t in block_ids])
    m = torch.cat([t.reshape(-1).to(torch.float64).cpu() for t in block_max])
    b_new = (V - 1) // block
    keep = (i >= 0) & (i < nb) & (i != b_new)
    i, m = i[keep], m[keep]
    order = torch.sort(i, stable=True).indices               # block id ascending ...
    i, m = i[order], m[order]
    order = torch.sort(-m, stable=True).indices              # ... then block max descending
    best = i[order][: n_keep - 1]
    out[: best.numel() + 1] = torch.sort(torch.cat([best, torch.tensor([b_new])])).values
    return out


def merge_attention(outs: Sequence[torch.Tensor], lses: Sequence[torch.Tensor],
                    sink: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Combine partial attention results over disjoint key sets, each computed
    without the sink: o = sum_r exp(lse_r - L) o_r, L = log(sum_r exp(lse_r) + exp(sink))."""
    L = torch.stack([t.to(torch.float64) for t in lses])                 # [P, H]
    O = torch.stack([t.to(torch.float64) for t in outs])                 # [P, H, c]
    s = torch.full_like(L[0], float("-inf")) if sink is None else sink.to(torch.float64)
    mx = torch.maximum(L.max(dim=0).values, s)
    den = torch.exp(L - mx).sum(dim=0) + torch.exp(s - mx)
    tot = mx + torch.log(den)
    w = torch.exp(L - tot)
    return (w.unsqueeze(-1) * O).sum(dim=0), tot


# ----------------------------------------------------------------------------------
# One rank's share of the pooled decode step, through the library
# ----------------------------------------------------------------------------------

@dataclass
class RankSelection:
    """What one rank contributes to the all-gather, per query ([B, Q, ...]):
    its pool as global block ids with their block maxima, and its top-k as global
    entry ids with their scores (-1 / -inf padded)."""
    pool_ids: torch.Tensor
    pool_max: torch.Tensor
    top_ids: torch.Tensor
    top_scores: torch.Tensor


def rank_select(qI, w, kI_local, lo: int, n_visible: torch.Tensor, k: int = 512, block: int = 8,
                n_keep: int = 2048) -> RankSelection:
    """The selection half of a Full-mode decode step on the entries [lo, lo + N_r)
    that this rank holds (kI_local = those rows, [B, N_r, ...]): full scan with the
    block max, the rank's own pool, rescoring of its candidates and its top-k with
    scores (csa2_topk's out_score).  Every step runs in the library; this function
    only shifts ids by the rank's offset.  lo must be a multiple of `block`."""
    if lo % block:
        raise ValueError("a rank's first entry must start a pool block")
    from . import pipeline as P
    B, Q = n_visible.shape
    N_r = kI_local.shape[1]
    nv = (n_visible - lo).clamp(0, N_r).contiguous()
    qI = P.mxfp4_query(qI, kI_local)
    nb = (N_r + block - 1) // block
    dev = n_visible.device
    bmax = C.alloc((B, Q, nb), dtype=torch.float32, device=dev)
    C.csa2_index_score(qI, w, kI_local, nv, block=block, want_scores=False, want_block_max=True, block_max=bmax)
    pool = C.alloc((B, Q, n_keep), dtype=torch.int32, device=dev)
    C.csa2_block_pool(bmax, nv, block=block, n_keep=n_keep, out=pool)
    sc, _ = C.csa2_index_score(qI, w, kI_local, nv, pool=pool, block=block)
    ids, top_sc = C.csa2_topk(sc, nv, k, pool=pool, block=block, want_scores=True)
    valid = pool >= 0
    pool_max = torch.gather(bmax, 2, pool.clamp_min(0).to(torch.int64))
    return RankSelection(
        pool_ids=torch.where(valid, pool.to(torch.int64) + lo // block, -1),
        pool_max=torch.where(valid, pool_max, torch.full_like(pool_max, float("-inf"))),
        top_ids=torch.where(ids >= 0, ids.to(torch.int64) + lo, -1),
        top_scores=top_sc)


def merge_selections(parts: Sequence[RankSelection], n_visible: torch.Tensor, k: int = 512, block: int = 8,
                     n_keep: int = 2048) -> Tuple[torch.Tensor, torch.Tensor]:
    """Merge the gathered per-rank selections of every query: (pool [B, Q, n_keep],
    top-k [B, Q, k]) as global ids, equal to the unsharded step's."""
    B, Q = n_visible.shape
    pool = torch.empty((B, Q, n_keep), dtype=torch.int64)
    top = torch.empty((B, Q, k), dtype=torch.int64)
    for b in range(B):
        for q in range(Q):
            V = int(n_visible[b, q])
            pool[b, q] = merge_pool([p.pool_ids[b, q] for p in parts], [p.pool_max[b, q] for p in parts], V, block,
                                    n_keep)
            top[b, q] = merge_topk([p.top_ids[b, q].cpu() for p in parts], [p.top_scores[b, q].cpu() for p in parts],
                                   k)
    return pool, top


def rank_attention(q, kv_local, lo: int, top_ids: torch.Tensor, swa, q_pos, with_window: bool,
                   window: int = 128, swa_pos0: int = 0, flags: int = C.ATTN_DEFAULT):
    """This rank's partial attention: over the selected entries it holds (global
    ids in [lo, lo + N_r)), plus the window on the one rank that owns it, without
    the sink.  Returns (o [B, Q, H, c] f32, lse [B, Q, H]) for merge_attention."""
    N_r = kv_local.shape[1]
    ids = top_ids.to(q.device)
    mine = (ids >= lo) & (ids < lo + N_r)
    idx = torch.where(mine, ids - lo, -1).to(torch.int32).contiguous()
    return C.csa2_sparse_attn(q, kv_local, idx, swa if with_window else None, q_pos, None,
                              window=window if with_window else 0, swa_pos0=swa_pos0, flags=flags,
                              out_dtype=torch.float32, want_lse=True)
