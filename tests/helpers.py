"""Comparison helpers shared by the GPU parity tests."""
import math
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


def valid_topk_sets(scores, cand, k, rms, rel_eps=1e-5, limit=64):
    """Every index set that the tie-window rule accepts as a top-k of the
    candidate ids `cand` under the oracle's scores: all candidates scoring above
    the window around the oracle's k-th score, plus any choice of the remaining
    count among the window's members (|score - kth| <= rel_eps * rms).  Each set
    is ascending and -1 padded to k.  These are the results that are equally
    correct; the list is built from the oracle's scores alone.  Returns None when
    the window allows more than `limit` sets."""
    import itertools
    cand = np.asarray(cand, dtype=np.int64)
    s = np.asarray(scores, dtype=np.float64)[cand]
    n = min(k, cand.shape[0])
    out_pad = np.full(k, -1, dtype=np.int64)
    if n == 0:
        return [out_pad]
    kth = np.sort(s)[::-1][n - 1]
    eps = rel_eps * rms
    above = cand[s > kth + eps]
    window = cand[np.abs(s - kth) <= eps]
    need = n - above.shape[0]
    if math.comb(window.shape[0], need) > limit:
        return None
    sets = []
    for comb in itertools.combinations(window.tolist(), need):
        sel = np.sort(np.concatenate([above, np.asarray(comb, dtype=np.int64)]))
        o = out_pad.copy()
        o[:n] = sel
        sets.append(o)
    return sets


def check_step_attention(gpu_out, gpu_idx, sets, oracle_attn, tol, what):
    """Check the attention a whole step produced (gpu_out, computed on the step's
    own selection gpu_idx) against the oracle.  `sets` are the equally correct
    selections the oracle enumerates (valid_topk_sets); the step's selection must
    be one of them (topk_swaps has checked that), and its output must match the
    oracle's attention over that set: oracle_attn(set) -> [H, c]."""
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    assert sets is not None, f"{what}: tie window too wide to enumerate the valid selections"
    match = [s for s in sets if np.array_equal(s, gpu_idx)]
    assert match, f"{what}: the step's selection is none of the oracle's valid selections"
    assert_close(gpu_out, oracle_attn(match[0]), tol, what)
    return len(sets)


def assert_exact_grid_scores(qI, w, KI, V, p):
    """Exact-grid precondition: every term w_h q_hd K_sd is a multiple of 2^-p and
    the magnitudes of one score's terms total less than 2^(24-p), so every partial
    sum is exact in fp32 in any order (and so equal to the f64 result)."""
    qI = np.asarray(qI, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    K = np.asarray(KI, dtype=np.float64)[:V]
    tot = np.abs(K) @ np.abs(qI).T @ np.abs(w)                 # [V]
    assert tot.max() < 2.0 ** (24 - p), f"term sums up to {tot.max()} exceed 2^{24 - p}"


GUARD_BYTES = 4096          # keeps the 256-byte alignment of the allocation it sits in
GUARD_FILL = 0xA5


class GuardedAlloc:
    """Stand-in for the binding's allocator in the GPU tests: every buffer the
    binding (or pipeline.py) allocates sits between two guard regions filled with
    GUARD_FILL, and verify() checks on the host that no call wrote outside its
    buffer.  Only buffers still alive are checked (a freed one may be reused)."""

    def __init__(self):
        import weakref
        self._weakref = weakref
        self.live = []
        self.checked = 0

    def alloc(self, shape, dtype, device):
        shape = (int(shape),) if isinstance(shape, int) else tuple(int(s) for s in shape)
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((GUARD_BYTES + n + GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8, device=device)
        view = raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)
        view._guard_raw = raw                        # the whole allocation lives as long as the view
        self.live.append((self._weakref.ref(view), n))
        return view

    def verify(self, what=""):
        keep, bad = [], []
        if any(r() is not None and r().is_cuda for r, _ in self.live):
            torch.cuda.synchronize()
        for r, n in self.live:
            v = r()
            if v is None:
                continue
            keep.append((r, n))
            raw = v._guard_raw
            head, tail = raw[:GUARD_BYTES], raw[GUARD_BYTES + n:]
            if not (bool((head == GUARD_FILL).all()) and bool((tail == GUARD_FILL).all())):
                bad.append((tuple(v.shape), v.dtype))
            self.checked += 1
        self.live = keep
        assert not bad, f"{what}: a call wrote outside its buffer(s) {bad}"
