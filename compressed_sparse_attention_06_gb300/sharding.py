"""Host-side logic for running the path on several GPUs (one process per GPU).

Two ways to split the work, neither needing a data-path collective for the first:

* by sequence (what bench.py does under torchrun): rank r owns sequences
  [r*B, (r+1)*B); every rank runs the whole step on its own sequences and the
  job's time is the maximum over ranks (weak scaling);
* by entry range, for one very long sequence: rank r scans entries [lo_r, hi_r),
  keeps its own top-k (global ids + scores) and attends over its share of the
  selected rows without the sink, returning (o_r, lse_r).  One all-gather of the
  small per-rank results then gives the exact answer: the top-k of the union of
  per-rank top-k lists in the (score desc, id asc) order, and the log-sum-exp
  combination of the partial attention outputs with the sink added once.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch


def sequences_for_rank(rank: int, world: int, per_rank: int) -> Tuple[int, int]:
    """(first global sequence index, count) owned by `rank`."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return rank * per_rank, per_rank


def entry_range(rank: int, world: int, n_entries: int) -> Tuple[int, int]:
    """Contiguous entry range [lo, hi) of `rank`, split as evenly as possible."""
    base, extra = divmod(n_entries, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


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
