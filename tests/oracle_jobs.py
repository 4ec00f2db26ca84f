"""Oracle work for the full-size parity tests, run in worker processes.

The 1M-entry FP4 workloads need the oracle's MXFP4 pack, unpack and scores of
every sequence (tens of seconds each in numpy), so the tests hand one sequence
per job to a process pool.  Workers draw the float rows themselves on the CPU with
the seeded input generators and return what the parent compares against the
GPU: the oracle's packed cache bytes and its scores.  Nothing here touches the
GPU or the CUDA library.

The pool uses the 'spawn' start method: a worker forked from a process that has
already used CUDA can hang.
"""
from __future__ import annotations

import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _torch_threads():
    import torch
    torch.set_num_threads(2)
    return torch


def fp4_decode_sequence(b: int, N: int, V: int, grid: bool, ki_new_row: np.ndarray, qI: np.ndarray,
                        w: np.ndarray, chunk: int = 1 << 18):
    """Sequence b of the FP4 decode workload through the oracle: MXFP4 pack of its
    indexer-key rows (the new token's row at position N-1 replaced by ki_new_row),
    the MXFP4 pack of the query, and the scores of the V visible entries.

    Returns (packed key rows [N, 68] uint8, packed query [H_I, 68] uint8, scores [N])."""
    _torch_threads()
    from compressed_sparse_attention_06_gb300 import workloads as W
    from oracle import csa2_oracle as O
    parts = []
    for r0 in range(0, N, chunk):
        n = min(chunk, N - r0)
        x = (W.fp4_grid_rows(GRID_KEY_SEED, b, r0, n, 128, "cpu") if grid
             else W.fp4_rows("KI", b, r0, n, N, "cpu"))
        parts.append(O.mxfp4_pack(x.numpy()))
    ki_ref = np.concatenate(parts)
    if ki_new_row is not None:
        ki_ref[N - 1] = O.mxfp4_pack(np.asarray(ki_new_row, dtype=np.float32).reshape(1, -1))[0]
    qI_ref = O.mxfp4_pack(np.asarray(qI, dtype=np.float32))
    sc = O.index_score(O.mxfp4_unpack(qI_ref), np.asarray(w, dtype=np.float64), O.mxfp4_unpack(ki_ref[:V]), V)
    return ki_ref, qI_ref, sc


# stream seed of the exact-grid indexer keys (one stream per sequence)
GRID_KEY_SEED = 4013


def pool(n_jobs: int) -> ProcessPoolExecutor:
    """A spawn-started process pool with small BLAS / torch thread counts per worker."""
    return ProcessPoolExecutor(max_workers=max(1, min(n_jobs, (os.cpu_count() or 2) // 2)),
                               mp_context=multiprocessing.get_context("spawn"))


def submit_all(ex: ProcessPoolExecutor, fn, arg_list):
    """Submit every job with BLAS threads per worker capped (workers start during the
    submits and inherit the environment of that moment)."""
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "2"
    try:
        return [ex.submit(fn, *args) for args in arg_list]
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
