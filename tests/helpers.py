"""Comparison helpers shared by the GPU parity tests."""
import numpy as np
import torch

from oracle import csa2_oracle as O


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy() if t.dtype != torch.uint8 and t.dtype not in (
        torch.int32, torch.int64) else t.detach().to("cpu").numpy()


def assert_close(g, o, tol, what=""):
    """|g - o| <= tol * (|o| + rms(o)) elementwise (the parity rule for floats)."""
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    fin = np.isfinite(o)
    assert np.array_equal(np.isfinite(g), fin), f"{what}: finite pattern differs"
    assert np.array_equal(g[~fin], o[~fin]), f"{what}: non-finite values differ"
    if not fin.any():
        return
    rms = np.sqrt(np.mean(o[fin] ** 2))
    err = np.abs(g[fin] - o[fin])
    bound = tol * (np.abs(o[fin]) + rms)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tol {tol}; worst err "
                           f"{err.max():.3e} (rms {rms:.3e})")


def topk_swaps(gpu_ids, oracle_scores, V, k, rel_eps=1e-5):
    """Compare a GPU top-k with the oracle's.  Indices must match exactly except
    for swaps whose oracle scores lie within eps = rel_eps * rms(I) of the oracle's
    k-th score.  Returns the number of such swaps; raises on any other difference."""
    gpu = [int(i) for i in np.asarray(gpu_ids) if i >= 0]
    ref = O.topk(oracle_scores, V, k)
    ref = [int(i) for i in ref if i >= 0]
    assert len(gpu) == len(ref), f"count {len(gpu)} vs {len(ref)}"
    assert gpu == sorted(gpu), "GPU ids not ascending"
    if gpu == ref:
        return 0
    s = np.asarray(oracle_scores, dtype=np.float64)[:V]
    kth = np.sort(s)[::-1][min(k, V) - 1]
    eps = rel_eps * np.sqrt(np.mean(s ** 2))
    diff = set(gpu) ^ set(ref)
    for i in diff:
        assert abs(s[i] - kth) <= eps, f"id {i}: score {s[i]} vs k-th {kth} (eps {eps})"
    return len(diff) // 2


def pool_swaps(gpu_pool, oracle_bmax, V, block, n_keep, rel_eps=1e-5):
    gpu = [int(b) for b in np.asarray(gpu_pool) if b >= 0]
    ref = [int(b) for b in O.block_pool(oracle_bmax, V, block, n_keep) if b >= 0]
    assert len(gpu) == len(ref)
    if gpu == ref:
        return 0
    bm = np.asarray(oracle_bmax, dtype=np.float64)
    b_new = (V - 1) // block
    assert b_new in gpu
    others = np.array([bm[b] for b in range(len(bm)) if b != b_new])
    kth = np.sort(others)[::-1][n_keep - 2]
    eps = rel_eps * np.sqrt(np.mean(bm ** 2))
    for b in set(gpu) ^ set(ref):
        assert abs(bm[b] - kth) <= eps, f"block {b}: {bm[b]} vs {kth}"
    return len(set(gpu) ^ set(ref)) // 2
