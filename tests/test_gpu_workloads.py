"""Whole-path parity on the five workloads at their full sizes, in the launch
configuration bench.py times (the same step functions and output dtypes), against
the oracle on every query of the decode workloads and on 256 seeded queries
(the first and the last among them) of the prefill chunk.

Two levels:

* Gaussian inputs (the workloads as written).  Scores within 1e-5 of the
  oracle's; selections equal the oracle's except for swaps whose oracle scores
  lie within 1e-5*rms of the k-th score (topk_swaps); the attention the step
  itself produced is compared with the oracle's attention over the step's
  selection, which must be one of the equally correct selections the oracle
  enumerates from its own scores (valid_topk_sets).  The attention kernel is
  also run once more on the oracle's own selection.
* Exact-grid inputs (indexer query, keys and weights snapped to a grid on which
  every product and partial sum is exact in fp32): scores, block maxima, pool and
  selections must equal the oracle's bit for bit, with no tie window.
"""
import math

import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import pipeline as P
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests import oracle_jobs as J
from tests.helpers import (assert_close, assert_exact_grid_scores, check_step_attention, pool_swaps, to_np,
                           topk_swaps, valid_topk_sets)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    yield
    C.csa2_ctx_check()
    torch.cuda.empty_cache()


def _np(t):
    return t.double().cpu().numpy()


def _rms(sc, V):
    return math.sqrt(float(np.mean(np.asarray(sc[:V], dtype=np.float64) ** 2))) if V else 0.0


class _RowMap:
    """Row lookup for the oracle when only the selected rows are materialised
    (rows are made on first use by `make`)."""

    def __init__(self, make):
        self.make = make
        self.rows = {}

    def __getitem__(self, s):
        s = int(s)
        if s not in self.rows:
            self.rows[s] = self.make(s)
        return self.rows[s]


def _gpu_attn_one(q, kv, ref_idx, swa, t, sink, swa_pos0=0, window=128):
    """GPU attention of one query ([H, c] slice of q), one sequence, given indices."""
    idx = torch.tensor(np.asarray(ref_idx), dtype=torch.int32, device=DEV).view(1, 1, -1)
    pos = torch.tensor([[t]], dtype=torch.int64, device=DEV)
    out, _ = C.csa2_sparse_attn(q.reshape(1, 1, *q.shape[-2:]).contiguous(), kv.unsqueeze(0).contiguous()
                                if kv.dim() == 2 else kv, idx, swa.unsqueeze(0).contiguous(), pos, sink,
                                window=window, swa_pos0=swa_pos0, out_dtype=torch.float32)
    return to_np(out)[0, 0]


def _check_selection(what, sc, V, gpu_idx, k, gpu_pool=None, gpu_bmax=None, n_keep=2048, exact=False):
    """Selection checks of one query against the oracle's scores sc; returns the
    valid selections (for the step's attention check)."""
    bm = O.block_max(sc, V, 8) if (gpu_bmax is not None or gpu_pool is not None) else None
    if gpu_bmax is not None:
        if exact:
            np.testing.assert_array_equal(gpu_bmax[: len(bm)], bm, err_msg=f"{what}: block max")
        else:
            assert_close(gpu_bmax[: len(bm)], bm, 1e-5, f"{what}: block max")
    if gpu_pool is not None:
        if exact:
            np.testing.assert_array_equal(gpu_pool, O.block_pool(bm, V, 8, n_keep), err_msg=f"{what}: pool")
        else:
            pool_swaps(gpu_pool, bm, V, 8, n_keep)
        cand = set(O.pool_candidates(gpu_pool, V).tolist())
        assert set(int(i) for i in gpu_idx if i >= 0) <= cand, f"{what}: top-k outside the pool"
    if exact:
        np.testing.assert_array_equal(gpu_idx, O.topk(sc, V, k), err_msg=f"{what}: top-k")
        return [O.topk(sc, V, k)]
    topk_swaps(gpu_idx, sc, V, k)
    return valid_topk_sets(sc, np.arange(V), k, _rms(sc, V))


def test_tiny_full_layer_end_to_end():
    """fp32 tiny layer: compressor (m=2, NORM+ROPE) -> indexer (8 heads) -> top-512 ->
    attention (16 heads, 128 window), all four queries at 4095..4092."""
    wl = W.tiny_full_layer(DEV)
    kv = C.csa2_compress(wl["Ca"], wl["Za"], wl.m, ba=wl["Ba"], flags=C.W_NORM | C.W_ROPE, out_fmt="f32")
    E = O.compress(_np(wl["Ca"]), _np(wl["Za"]), wl.m, _np(wl["Ba"]))
    kv_ref = O.compress_write(E, O.NORM_W | O.ROPE_W, wl.m, 0)
    assert_close(to_np(kv), kv_ref, 1e-4, "compressed entries")
    nv = P.visible_entries(wl.q_pos, wl.m)
    sc, idx = P.full_topk_step(wl["qI"], wl["w"], wl["KI"], nv)
    out, _ = C.csa2_sparse_attn(wl["q"], kv.unsqueeze(0), idx, wl["swa"], wl.q_pos, wl["sink"], out_dtype=torch.float32)
    for qi, t in enumerate(wl.q_pos[0].tolist()):
        V = t // 2
        ref_sc = O.index_score(_np(wl["qI"][0, qi]), _np(wl["w"][0, qi]), _np(wl["KI"][0]), V)
        assert_close(to_np(sc)[0, qi], ref_sc, 1e-4, f"scores q{qi}")
        sets = _check_selection(f"q{qi}", ref_sc, V, to_np(idx)[0, qi], 512)
        ref_idx = O.topk(ref_sc, V, 512)

        def attn(sel, qi=qi, t=t):
            return O.sparse_attn(_np(wl["q"][0, qi]), kv_ref, sel, _np(wl["swa"][0]), 0, t, _np(wl["sink"]), 128)[0]
        g = _gpu_attn_one(wl["q"][0, qi], kv, ref_idx, wl["swa"][0], t, wl["sink"])
        assert_close(g, attn(ref_idx), 1e-4, f"attention q{qi}")
        check_step_attention(to_np(out)[0, qi], to_np(idx)[0, qi], sets, attn, 1e-4, f"step attention q{qi}")


# ------------------------------------------------------------------ FP4 decode at 1M (headline)
def _fp4_caches(B, N, grid=False, seq0=0):
    kv = torch.empty((B, N, 288), dtype=torch.uint8, device=DEV)
    ki = torch.empty((B, N, 68), dtype=torch.uint8, device=DEV)
    ch = 1 << 16
    for b in range(B):
        for r0 in range(0, N, ch):
            n = min(ch, N - r0)
            C.csa2_fp4_pack(W.fp4_rows("kv", seq0 + b, r0, n, N, DEV), C.FP4_E4M3x16, out=kv[b, r0:r0 + n])
            rows = (W.fp4_grid_rows(J.GRID_KEY_SEED, seq0 + b, r0, n, 128, DEV) if grid
                    else W.fp4_rows("KI", seq0 + b, r0, n, N, DEV))
            C.csa2_fp4_pack(rows, C.MXFP4_E8M0x32, out=ki[b, r0:r0 + n])
    return kv, ki


def _fp4_kv_row(b, N):
    return lambda s: O.nvfp4_unpack(O.nvfp4_pack(W.fp4_rows("kv", b, s, 1, N, "cpu").numpy()))[0]


def _run_fp4_decode(B, N, H, k, grid):
    """The bench's FP4 decode step (new-token rows, query pack, full scan with scores,
    block maxima and their histogram, pool + top-k, attention into bf16), then every
    sequence through the oracle."""
    wl = W.fp4_decode(DEV, B=B, N=N, H=H, grid=grid)
    kv, ki = _fp4_caches(B, N, grid)
    t = N - 1
    V = t
    # the oracle's per-sequence work starts first (spawned workers, CPU only)
    ex = J.pool(B)
    futs = J.submit_all(ex, J.fp4_decode_sequence,
                        [(b, N, V, grid, None if grid else wl["KI_new"][b].float().cpu().numpy(),
                          wl["qI"][b, 0].float().cpu().numpy(), wl["w"][b, 0].cpu().numpy()) for b in range(B)])
    # the step, as bench.py runs it: the new token's cache rows, then the layer
    if not grid:
        C.csa2_compress(wl["C_new"], wl["Z_new"], 1, pos0=wl.q_pos[:, 0].clone(), flags=C.W_ROPE, out=kv[:, t],
                        out_seq_stride=N)
        C.csa2_fp4_pack(wl["KI_new"].reshape(B, 128), C.MXFP4_E8M0x32, out=ki[:, t], out_ld=N * 68)
    sink = wl["sink"] if H == 64 else W.normal_tensor((H,), 4109, 0, torch.float32, DEV)
    nv = P.visible_entries(wl.q_pos, 1)
    buf = P.alloc_decode(B, 1, N, H, 512, DEV, out_dtype=torch.bfloat16, k=k)
    # as bench.py runs it: the attention's query half on a second stream beside the selection
    P.full_decode_step(wl["qI"], wl["w"], ki, wl["q"], kv, wl["swa"], wl.q_pos, nv, sink, buf, k=k,
                       side_stream=torch.cuda.Stream())
    C.csa2_ctx_check()
    n_sets = []
    for b in range(B):
        what = f"{'grid ' if grid else ''}b{b}"
        ki_ref, qI_ref, sc = futs[b].result()
        np.testing.assert_array_equal(to_np(ki[b]), ki_ref, err_msg=f"{what}: MXFP4 cache bytes")
        np.testing.assert_array_equal(to_np(buf.qI_mx[b, 0]), qI_ref, err_msg=f"{what}: MXFP4 query bytes")
        if not P.pool_topk_applies(k, 8, 2048, buf.block_max.shape[-1]):
            # top-1024: the step rescored its best blocks with the candidate scan
            tb = to_np(buf.top_blocks[b, 0]).astype(np.int64)
            ids = (tb[:, None] * 8 + np.arange(8)).reshape(-1)
            ok = np.repeat(tb >= 0, 8) & (ids < V)
            assert ok.sum() >= k
            assert_close(to_np(buf.cand_scores[b, 0])[ok], sc[ids[ok]], 1e-5, f"{what}: best blocks' scores")
        elif grid:
            assert_exact_grid_scores(O.mxfp4_unpack(qI_ref), _np(wl["w"][b, 0]), O.mxfp4_unpack(ki_ref), V, 3)
            np.testing.assert_array_equal(to_np(buf.scores[b, 0])[:V], sc[:V], err_msg=f"{what}: scores")
        else:
            assert_close(to_np(buf.scores[b, 0])[:V], sc[:V], 1e-5, f"{what}: scores")
        sets = _check_selection(what, sc, V, to_np(buf.idx[b, 0]), k, to_np(buf.pool[b, 0]),
                                to_np(buf.block_max[b, 0]), exact=grid)
        rows = _RowMap(_fp4_kv_row(b, N))

        def attn(sel, b=b):
            return O.sparse_attn(_np(wl["q"][b, 0]), rows, sel, _np(wl["swa"][b]), 0, t, _np(sink), 128)[0]
        n_sets.append(check_step_attention(to_np(buf.out[b, 0]), to_np(buf.idx[b, 0]), sets, attn, 2e-2,
                                           f"{what}: step attention"))
        ref_idx = O.topk(sc, V, k)
        g = _gpu_attn_one(wl["q"][b, 0], kv[b], ref_idx, wl["swa"][b], t, sink)
        assert_close(g, attn(ref_idx), 2e-2, f"{what}: attention on the oracle's selection")
        if not grid:
            # the new token's main-KV row: RoPE'd copy of C_new (m = 1), FP4-packed
            new_ref = O.compress_write(_np(wl["C_new"][b]), O.ROPE_W, 1, t)
            got = O.nvfp4_unpack(to_np(kv[b, t:t + 1]))[0]
            ref = O.nvfp4_unpack(O.nvfp4_pack(new_ref.astype(np.float32)))[0]
            s = np.repeat(O.e4m3_decode(to_np(kv[b, t, 256:])), 16)
            assert np.all(np.abs(got - ref) <= 2 * s + 1e-6)
    ex.shutdown()
    return n_sets


def test_fp4_decode_1M_full_size_all_8_sequences():
    """FP4-cache decode at 1M context, batch 8, exactly as bench.py runs it (bf16
    output); all 8 sequences through the oracle."""
    _run_fp4_decode(8, 1 << 20, 64, 512, grid=False)


def test_fp4_decode_1M_exact_grid_all_8_sequences():
    """The headline step on exact-grid indexer inputs (E2M1 values with block scale
    2^0, weights on multiples of 1/2): block maxima, pool and top-512 bit-exact for
    all 8 sequences, with no tie window."""
    _run_fp4_decode(8, 1 << 20, 64, 512, grid=True)


def test_fp4_decode_v4pro_variant_all_4_sequences():
    """The V4-Pro configuration (DSA-to-CSA/HCA page, «两个已公开配置»): CSA top-1024,
    128 query heads (two 64-head tensor-core passes over the same selected rows),
    64 indexer heads; FP4 caches, 4 sequences of 262,144 entries, all through the
    oracle."""
    _run_fp4_decode(4, 1 << 18, 128, 1024, grid=False)


# ------------------------------------------------------------------ bf16 decode at 64K
def _run_decode_bf16(grid):
    wl = W.decode_full_bf16(DEV, grid=grid)
    B, N = wl.B, wl.N
    nv = P.visible_entries(wl.q_pos, 1)
    buf = P.alloc_decode(B, 1, N, 64, 512, DEV)                  # bf16 output, as bench.py
    P.full_decode_step(wl["qI"], wl["w"], wl["KI"], wl["q"], wl["kv"], wl["swa"], wl.q_pos, nv, wl["sink"], buf)
    C.csa2_ctx_check()
    t = N - 1
    V = N - 1
    for b in range(B):
        what = f"{'grid ' if grid else ''}b{b}"
        K_np = _np(wl["KI"][b])
        qI, w = _np(wl["qI"][b, 0]), _np(wl["w"][b, 0])
        sc = O.index_score(qI, w, K_np, V)
        # the step's full scan scores (the top-k reads its best blocks' entries from them)
        if grid:
            assert_exact_grid_scores(qI, w, K_np, V, 7)
            np.testing.assert_array_equal(to_np(buf.scores[b, 0])[:V], sc[:V], err_msg=f"{what}: scores")
        else:
            assert_close(to_np(buf.scores[b, 0])[:V], sc[:V], 1e-5, f"{what}: scores")
        sets = _check_selection(what, sc, V, to_np(buf.idx[b, 0]), 512, to_np(buf.pool[b, 0]),
                                to_np(buf.block_max[b, 0]), exact=grid)
        if not grid:
            planted = to_np(wl["planted"][b])
            mu, sd = sc[:4096].mean(), sc[:4096].std()
            assert np.all(sc[planted] >= mu + 8 * sd)
            assert set(planted.tolist()) <= set(to_np(buf.idx[b, 0]).tolist())
            assert set((planted // 8).tolist()) <= set(to_np(buf.pool[b, 0]).tolist())
        rows = _RowMap(lambda s, b=b: _np(wl["kv"][b, s]))

        def attn(sel, b=b):
            return O.sparse_attn(_np(wl["q"][b, 0]), rows, sel, _np(wl["swa"][b]), 0, t, _np(wl["sink"]), 128)[0]
        check_step_attention(to_np(buf.out[b, 0]), to_np(buf.idx[b, 0]), sets, attn, 2e-2, f"{what}: step attention")
        ref_idx = O.topk(sc, V, 512)
        g = _gpu_attn_one(wl["q"][b, 0], wl["kv"][b], ref_idx, wl["swa"][b], t, wl["sink"])
        assert_close(g, attn(ref_idx), 2e-2, f"{what}: attention on the oracle's selection")


def _cand_slots(pool_row, V, block=8):
    """Positions, in a candidate-score row, of the visible candidates in ascending
    entry order (candidate c is entry pool[c // block] * block + c % block)."""
    p = pool_row.cpu().numpy().astype(np.int64)
    ent = (p[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    ok = (np.repeat(p, block) >= 0) & (ent < V)
    slots = np.nonzero(ok)[0]
    return slots[np.argsort(ent[slots], kind="stable")]


def test_decode_full_bf16_64k_full_size_all_32_sequences():
    """Decoder Full-mode decode, bf16, batch 32 x 64K, with the pool; all 32
    sequences; the 16 planted keys score >= mu + 8 sigma and are selected."""
    _run_decode_bf16(grid=False)


def test_decode_full_bf16_64k_exact_grid_all_32_sequences():
    """The 64K bf16 decode step on exact-grid indexer inputs: block maxima, pool,
    candidate scores and top-512 bit-exact for all 32 sequences."""
    _run_decode_bf16(grid=True)


# ------------------------------------------------------------------ Reindex + 3 Reuse at 256K
def _run_reindex(grid):
    wl = W.reindex_reuse_bf16(DEV, grid=grid)
    B, N = wl.B, wl.N
    nv = P.visible_entries(wl.q_pos, 1)
    cand_scores = torch.empty((B, 1, 16384), dtype=torch.float32, device=DEV)
    idx = P.reindex_step(wl["qI"], wl["w"], wl["KI"], wl["pool"], nv, cand_scores=cand_scores)
    outs = [P.reuse_attention(wl[f"q{l}"], wl["kv"], idx, wl[f"swa{l}"], wl.q_pos, wl["sink"]) for l in range(4)]
    C.csa2_ctx_check()
    t = N - 1
    V = N - 1
    for b in range(B):
        what = f"{'grid ' if grid else ''}b{b}"
        qI, w = _np(wl["qI"][b, 0]), _np(wl["w"][b, 0])
        K_np = _np(wl["KI"][b])
        full = O.index_score(qI, w, K_np, V)
        pool = to_np(wl["pool"][b, 0])
        cand = O.pool_candidates(pool, V)
        gpu = to_np(idx[b, 0])
        ref = O.reindex_topk(full, pool, V, 512)
        cs = to_np(cand_scores[b, 0]).reshape(-1)[_cand_slots(wl["pool"][b, 0], V)]
        assert set(int(i) for i in gpu if i >= 0) <= set(cand.tolist())
        if grid:
            assert_exact_grid_scores(qI, w, K_np, V, 7)
            np.testing.assert_array_equal(cs, full[cand], err_msg=f"{what}: candidate scores")
            np.testing.assert_array_equal(gpu, ref, err_msg=f"{what}: top-512")
            sets = [ref]
        else:
            assert_close(cs, full[cand], 1e-5, f"{what}: candidate scores")
            sets = valid_topk_sets(full, cand, 512, _rms(full, V))
            kth = np.sort(full[cand])[::-1][511]
            eps = 1e-5 * _rms(full, V)
            for i in set(gpu.tolist()) ^ set(ref.tolist()):
                assert abs(full[i] - kth) <= eps, f"{what}: id {i} outside the tie window"
        rows = _RowMap(lambda s, b=b: _np(wl["kv"][b, s]))
        for l in range(4):
            def attn(sel, b=b, l=l):
                return O.sparse_attn(_np(wl[f"q{l}"][b, 0]), rows, sel, _np(wl[f"swa{l}"][b]), 0, t,
                                     _np(wl["sink"]), 128)[0]
            check_step_attention(to_np(outs[l][b, 0]), gpu, sets, attn, 2e-2, f"{what}: layer {l} step attention")
            if l == 0:
                g = _gpu_attn_one(wl["q0"][b, 0], wl["kv"][b], ref, wl["swa0"][b], t, wl["sink"])
                assert_close(g, attn(ref), 2e-2, f"{what}: attention on the oracle's selection")


def test_reindex_reuse_bf16_256k_full_size_all_64_sequences():
    """Reindex over the pooled 16,384 candidates, top-512, then the Reindex layer and
    three Reuse layers attend with their own q and window; batch 64 x 256K, all 64
    sequences and all four layers' outputs through the oracle."""
    _run_reindex(grid=False)


def test_reindex_reuse_bf16_256k_exact_grid_all_64_sequences():
    """Reindex on exact-grid indexer inputs: candidate scores and top-512 bit-exact
    for all 64 sequences."""
    _run_reindex(grid=True)


# ------------------------------------------------------------------ prefill chunk
N_PREFILL_CHECKED = 256


def test_prefill_chunk_full_size_256_queries():
    """Encoder prefill chunk: 8192 queries on a 131,072-token context, overlapped
    compressor (m=4, carried state), 64-head indexer over up to 34,816 entries,
    top-512 per query, attention with sink (bf16 output, as bench.py); 256 seeded
    queries (the first and the last among them) through the oracle."""
    wl = W.prefill_chunk_bf16(DEV)
    N, Q, m = wl.N, wl.Q, wl.m
    nce = wl.meta["n_ctx_entries"]
    kv = torch.empty((1, N, 512), dtype=torch.bfloat16, device=DEV)
    kv[0, :nce] = wl["kv_ctx"][0]
    pos0 = torch.tensor([wl.meta["pos0"]], dtype=torch.int64, device=DEV)
    buf = P.alloc_prefill(Q, N, 64, 512, DEV, wl.q_pos, m, swa_cap=wl.meta["swa_cap"])
    P.prefill_chunk_step(wl["Ca"], wl["Cb"], wl["Za"], wl["Zb"], wl["Ba"], wl["Bb"], wl["prev_Cb"], wl["prev_Zb"],
                         kv, nce, pos0, m, wl["qI"], wl["w"], wl["KI"], wl["q"], wl["swa"], wl.meta["swa_pos0"],
                         wl.q_pos, wl["sink"], buf)
    C.csa2_ctx_check()
    # compressor: the new entries, against the oracle's overlapped compressor
    E = O.compress(_np(wl["Ca"]), _np(wl["Za"]), m, _np(wl["Ba"]), _np(wl["Cb"]), _np(wl["Zb"]), _np(wl["Bb"]),
                   _np(wl["prev_Cb"]), _np(wl["prev_Zb"]))
    new_ref = O.compress_write(E, O.NORM_W | O.ROPE_W, m, wl.meta["pos0"])
    assert_close(to_np(kv[0, nce:].float()), new_ref, 2e-2, "compressed chunk")
    kv_ref = np.concatenate([_np(wl["kv_ctx"][0]), new_ref])      # the oracle's own entries
    K_np = _np(wl["KI"][0])
    sample = W.distinct_sample(Q - 2, N_PREFILL_CHECKED - 2, 5101, 0, "cpu").numpy() + 1
    queries = [0] + sample.tolist() + [Q - 1]
    assert len(set(queries)) == N_PREFILL_CHECKED
    qsel = torch.tensor(queries, dtype=torch.int64, device=DEV)
    scores = to_np(buf.scores[0].index_select(0, qsel))
    idx = to_np(buf.idx[0].index_select(0, qsel))
    out = to_np(buf.out[0].index_select(0, qsel))
    for j, qi in enumerate(queries):
        t = int(wl.q_pos[0, qi])
        V = t // m
        sc = O.index_score(_np(wl["qI"][0, qi]), _np(wl["w"][0, qi]), K_np, V)
        assert_close(scores[j], sc, 1e-5, f"scores q{qi}")
        sets = _check_selection(f"q{qi}", sc, V, idx[j], 512)

        def attn(sel, qi=qi, t=t):
            return O.sparse_attn(_np(wl["q"][0, qi]), kv_ref, sel, _np(wl["swa"][0]), wl.meta["swa_pos0"], t,
                                 _np(wl["sink"]), 128)[0]
        check_step_attention(out[j], idx[j], sets, attn, 2e-2, f"q{qi}: step attention")
        if qi in (0, Q - 1):
            ref_idx = O.topk(sc, V, 512)
            g = _gpu_attn_one(wl["q"][0, qi], kv[0], ref_idx, wl["swa"][0], t, wl["sink"], wl.meta["swa_pos0"])
            assert_close(g, attn(ref_idx), 2e-2, f"attention on the oracle's selection q{qi}")


def test_dsa_token_level_top2048():
    """DSA-style selection (DSA-to-CSA/HCA page, the DSA baseline: top-2048 tokens,
    m = 1) and attention over the 2,048 selected rows plus the window, bf16, 64 heads."""
    B, N, k = 2, 100000, 2048
    qI = W.normal_tensor((B, 1, 64, 128), 4201, 0, torch.bfloat16, DEV)
    w = W.normal_tensor((B, 1, 64), 4202, 0, torch.float32, DEV)
    KI = W.normal_tensor((B, N, 128), 4203, 0, torch.bfloat16, DEV)
    kv = W.normal_tensor((B, N, 512), 4204, 0, torch.bfloat16, DEV)
    q = W.normal_tensor((B, 1, 64, 512), 4205, 0, torch.bfloat16, DEV)
    swa = W.normal_tensor((B, 128, 512), 4206, 0, torch.bfloat16, DEV)
    sink = W.normal_tensor((64,), 4207, 0, torch.float32, DEV)
    q_pos = torch.tensor([[N - 1], [61234]], dtype=torch.int64, device=DEV)
    nv = P.visible_entries(q_pos, 1)
    sc, idx = P.full_topk_step(qI, w, KI, nv, k=k)
    out, _ = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=128, out_dtype=torch.float32)
    C.csa2_ctx_check()
    for b in range(B):
        V = int(nv[b, 0])
        ref_sc = O.index_score(_np(qI[b, 0]), _np(w[b, 0]), _np(KI[b]), V)
        sets = _check_selection(f"b{b}", ref_sc, V, to_np(idx[b, 0]), k)
        kv_b = _np(kv[b])

        def attn(sel, b=b):
            return O.sparse_attn(_np(q[b, 0]), kv_b, sel, _np(swa[b]), 0, int(q_pos[b, 0]), _np(sink), 128)[0]
        check_step_attention(to_np(out[b, 0]), to_np(idx[b, 0]), sets, attn, 2e-2, f"b{b}: step attention")
        ref_idx = O.topk(ref_sc, V, k)
        g = _gpu_attn_one(q[b, 0], kv[b], ref_idx, swa[b], int(q_pos[b, 0]), sink)
        assert_close(g, attn(ref_idx), 2e-2, f"attention b{b}")
