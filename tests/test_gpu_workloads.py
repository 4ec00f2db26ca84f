"""Whole-path parity on the five workloads, at their full sizes and in the launch
configuration bench.py times, checked against the oracle on sampled sequences /
queries (the oracle computes those one by one).

Selection is compared by the tie-window rule (indices equal except swaps whose
oracle scores lie within 1e-5*rms of the k-th score).  Attention is compared on the
oracle's own indices: the GPU attention is run again with them, so no GPU output
ever becomes an oracle input."""
import math

import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import pipeline as P
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, pool_swaps, to_np, topk_swaps

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


class _RowMap:
    """Row lookup for the oracle when only the selected rows are materialised."""

    def __init__(self, rows):
        self.rows = rows

    def __getitem__(self, s):
        return self.rows[int(s)]


def _gpu_attn_one(q, kv, ref_idx, swa, t, sink, swa_pos0=0, window=128):
    """GPU attention of one query ([H, c] slice of q), one sequence, given indices."""
    idx = torch.tensor(np.asarray(ref_idx), dtype=torch.int32, device=DEV).view(1, 1, -1)
    pos = torch.tensor([[t]], dtype=torch.int64, device=DEV)
    out, _ = C.csa2_sparse_attn(q.reshape(1, 1, *q.shape[-2:]).contiguous(), kv.unsqueeze(0).contiguous()
                                if kv.dim() == 2 else kv, idx, swa.unsqueeze(0).contiguous(), pos, sink,
                                window=window, swa_pos0=swa_pos0, out_dtype=torch.float32)
    return to_np(out)[0, 0]


def test_tiny_full_layer_end_to_end():
    """fp32 tiny layer: compressor (m=2, NORM+ROPE) -> indexer (8 heads) -> top-512 ->
    attention (16 heads, 128 window), four queries at 4095..4092."""
    wl = W.tiny_full_layer(DEV)
    kv = C.csa2_compress(wl["Ca"], wl["Za"], wl.m, ba=wl["Ba"], flags=C.W_NORM | C.W_ROPE, out_fmt="f32")
    E = O.compress(_np(wl["Ca"]), _np(wl["Za"]), wl.m, _np(wl["Ba"]))
    kv_ref = O.compress_write(E, O.NORM_W | O.ROPE_W, wl.m, 0)
    assert_close(to_np(kv), kv_ref, 1e-4, "compressed entries")
    nv = P.visible_entries(wl.q_pos, wl.m)
    sc, idx = P.full_topk_step(wl["qI"], wl["w"], wl["KI"], nv)
    for qi, t in enumerate(wl.q_pos[0].tolist()):
        V = t // 2
        ref_sc = O.index_score(_np(wl["qI"][0, qi]), _np(wl["w"][0, qi]), _np(wl["KI"][0]), V)
        assert_close(to_np(sc)[0, qi], ref_sc, 1e-4, f"scores q{qi}")
        topk_swaps(to_np(idx)[0, qi], ref_sc, V, 512)
        ref_idx = O.topk(ref_sc, V, 512)
        o, _, _ = O.sparse_attn(_np(wl["q"][0, qi]), kv_ref, ref_idx, _np(wl["swa"][0]), 0, t, _np(wl["sink"]), 128)
        g = _gpu_attn_one(wl["q"][0, qi], kv, ref_idx, wl["swa"][0], t, wl["sink"])
        assert_close(g, o, 1e-4, f"attention q{qi}")


def _check_decode_query(b, V, qI, w, K_np, gpu_idx, gpu_pool, gpu_bmax, k=512, n_keep=2048):
    sc = O.index_score(qI, w, K_np, V)
    topk_swaps(gpu_idx, sc, V, k)
    if gpu_bmax is not None:
        bm = O.block_max(sc, V, 8)
        assert_close(gpu_bmax[: len(bm)], bm, 1e-5, f"block max b{b}")
    if gpu_pool is not None:
        pool_swaps(gpu_pool, O.block_max(sc, V, 8), V, 8, n_keep)
        cand = set(O.pool_candidates(gpu_pool, V).tolist())
        assert set(int(i) for i in gpu_idx if i >= 0) <= cand      # the top-k lies inside the pool
    return sc, O.topk(sc, V, k)


def test_fp4_decode_1M_full_size():
    """FP4-cache decode at 1M context, batch 8, exactly as bench.py runs it; sampled
    sequences 0 and 7 through the oracle."""
    B, N = 8, 1 << 20
    wl = W.fp4_decode(DEV, B=B, N=N)
    kv = torch.empty((B, N, 288), dtype=torch.uint8, device=DEV)
    ki = torch.empty((B, N, 68), dtype=torch.uint8, device=DEV)
    ch = 1 << 16
    for b in range(B):
        for r0 in range(0, N, ch):
            C.csa2_fp4_pack(W.fp4_rows("kv", b, r0, ch, N, DEV), C.FP4_E4M3x16, out=kv[b, r0:r0 + ch])
            C.csa2_fp4_pack(W.fp4_rows("KI", b, r0, ch, N, DEV), C.MXFP4_E8M0x32, out=ki[b, r0:r0 + ch])
    t = N - 1
    pos_new = wl.q_pos[:, 0].clone()
    C.csa2_compress(wl["C_new"], wl["Z_new"], 1, pos0=pos_new, flags=C.W_ROPE, out=kv[:, t], out_seq_stride=N)
    C.csa2_fp4_pack(wl["KI_new"].reshape(B, 128), C.MXFP4_E8M0x32, out=ki[:, t], out_ld=N * 68)
    nv = P.visible_entries(wl.q_pos, 1)
    buf = P.alloc_decode(B, 1, N, 64, 512, DEV, out_dtype=torch.float32)
    P.full_decode_step(wl["qI"], wl["w"], ki, wl["q"], kv, wl["swa"], wl.q_pos, nv, wl["sink"], buf)
    C.csa2_ctx_check()
    for b in (0, B - 1):
        ki_f = torch.cat([W.fp4_rows("KI", b, r0, ch, N, DEV) for r0 in range(0, N, ch)]).cpu().numpy()
        ki_ref = O.mxfp4_pack(ki_f)
        ki_ref[t] = O.mxfp4_pack(wl["KI_new"][b].float().cpu().numpy())[0]
        np.testing.assert_array_equal(to_np(ki[b]), ki_ref)            # cache bytes, bit-exact
        V = N - 1
        K_np = O.mxfp4_unpack(ki_ref[:V])
        # the FP4 QK path: the step packed qI to MXFP4 (bytes bit-exact with the oracle's pack)
        qI_ref = O.mxfp4_pack(wl["qI"][b, 0].float().cpu().numpy())
        np.testing.assert_array_equal(to_np(buf.qI_mx[b, 0]), qI_ref)
        _, ref_idx = _check_decode_query(b, V, O.mxfp4_unpack(qI_ref), _np(wl["w"][b, 0]), K_np,
                                         to_np(buf.idx[b, 0]), to_np(buf.pool[b, 0]), to_np(buf.block_max[b, 0]))
        rows = {int(s): O.nvfp4_unpack(O.nvfp4_pack(W.fp4_rows("kv", b, int(s), 1, N, "cpu").numpy()))[0]
                for s in ref_idx if s >= 0}
        o, _, _ = O.sparse_attn(_np(wl["q"][b, 0]), _RowMap(rows), ref_idx, _np(wl["swa"][b]), 0, t,
                                _np(wl["sink"]), 128)
        if np.array_equal(to_np(buf.idx[b, 0]), ref_idx):
            assert_close(to_np(buf.out[b, 0]), o, 2e-2, f"attention (pipeline) b{b}")
        g = _gpu_attn_one(wl["q"][b, 0], kv[b], ref_idx, wl["swa"][b], t, wl["sink"])
        assert_close(g, o, 2e-2, f"attention b{b}")
        # the new token's main-KV row: RoPE'd copy of C_new (m = 1), FP4-packed
        new_ref = O.compress_write(_np(wl["C_new"][b]), O.ROPE_W, 1, t)
        got = O.nvfp4_unpack(to_np(kv[b, t:t + 1]))[0]
        ref = O.nvfp4_unpack(O.nvfp4_pack(new_ref.astype(np.float32)))[0]
        s = np.repeat(O.e4m3_decode(to_np(kv[b, t, 256:])), 16)
        assert np.all(np.abs(got - ref) <= 2 * s + 1e-6)


def test_decode_full_bf16_64k_full_size():
    """Decoder Full-mode decode, bf16, batch 32 x 64K, with the pool; sampled
    sequences 0 and 31; the 16 planted keys score >= mu + 8 sigma and are selected."""
    wl = W.decode_full_bf16(DEV)
    B, N = wl.B, wl.N
    nv = P.visible_entries(wl.q_pos, 1)
    buf = P.alloc_decode(B, 1, N, 64, 512, DEV, out_dtype=torch.float32)
    P.full_decode_step(wl["qI"], wl["w"], wl["KI"], wl["q"], wl["kv"], wl["swa"], wl.q_pos, nv, wl["sink"], buf)
    C.csa2_ctx_check()
    t = N - 1
    for b in (0, B - 1):
        V = N - 1
        sc, ref_idx = _check_decode_query(b, V, _np(wl["qI"][b, 0]), _np(wl["w"][b, 0]), _np(wl["KI"][b]),
                                          to_np(buf.idx[b, 0]), to_np(buf.pool[b, 0]), to_np(buf.block_max[b, 0]))
        planted = to_np(wl["planted"][b])
        mu, sd = sc[:4096].mean(), sc[:4096].std()
        assert np.all(sc[planted] >= mu + 8 * sd)
        assert set(planted.tolist()) <= set(to_np(buf.idx[b, 0]).tolist())
        assert set((planted // 8).tolist()) <= set(to_np(buf.pool[b, 0]).tolist())
        rows = {int(s): _np(wl["kv"][b, int(s)]) for s in ref_idx if s >= 0}
        o, _, _ = O.sparse_attn(_np(wl["q"][b, 0]), _RowMap(rows), ref_idx, _np(wl["swa"][b]), 0, t,
                                _np(wl["sink"]), 128)
        g = _gpu_attn_one(wl["q"][b, 0], wl["kv"][b], ref_idx, wl["swa"][b], t, wl["sink"])
        assert_close(g, o, 2e-2, f"attention b{b}")
        if np.array_equal(to_np(buf.idx[b, 0]), ref_idx):
            assert_close(to_np(buf.out[b, 0]), o, 2e-2, f"attention (pipeline) b{b}")


def test_reindex_reuse_bf16_256k_full_size():
    """Reindex over the pooled 16,384 candidates, top-512, then the Reindex layer and
    three Reuse layers attend with their own q and window; batch 64 x 256K."""
    wl = W.reindex_reuse_bf16(DEV)
    B, N = wl.B, wl.N
    nv = P.visible_entries(wl.q_pos, 1)
    idx = P.reindex_step(wl["qI"], wl["w"], wl["KI"], wl["pool"], nv)
    outs = [P.reuse_attention(wl[f"q{l}"], wl["kv"], idx, wl[f"swa{l}"], wl.q_pos, wl["sink"]) for l in range(4)]
    C.csa2_ctx_check()
    t = N - 1
    for b in (0, B - 1):
        V = N - 1
        full = O.index_score(_np(wl["qI"][b, 0]), _np(wl["w"][b, 0]), _np(wl["KI"][b]), V)
        pool = to_np(wl["pool"][b, 0])
        ref = O.reindex_topk(full, pool, V, 512)
        gpu = to_np(idx[b, 0])
        cand = O.pool_candidates(pool, V)
        assert set(int(i) for i in gpu if i >= 0) <= set(cand.tolist())
        if not np.array_equal(gpu, ref):
            kth = np.sort(full[cand])[::-1][511]
            eps = 1e-5 * math.sqrt(np.mean(full[:V] ** 2))
            for i in set(gpu.tolist()) ^ set(ref.tolist()):
                assert abs(full[i] - kth) <= eps
        rows = {int(s): _np(wl["kv"][b, int(s)]) for s in ref if s >= 0}
        for l in range(4):
            o, _, _ = O.sparse_attn(_np(wl[f"q{l}"][b, 0]), _RowMap(rows), ref, _np(wl[f"swa{l}"][b]), 0, t,
                                    _np(wl["sink"]), 128)
            g = _gpu_attn_one(wl[f"q{l}"][b, 0], wl["kv"][b], ref, wl[f"swa{l}"][b], t, wl["sink"])
            assert_close(g, o, 2e-2, f"layer {l} b{b}")
            if np.array_equal(gpu, ref):
                assert_close(to_np(outs[l][b, 0].float()), o, 2e-2, f"layer {l} (pipeline) b{b}")


def test_prefill_chunk_full_size():
    """Encoder prefill chunk: 8192 queries on a 131,072-token context, overlapped
    compressor (m=4, carried state), 64-head indexer over up to 34,816 entries,
    top-512 per query, attention with sink; sampled queries through the oracle."""
    wl = W.prefill_chunk_bf16(DEV)
    N, Q, m = wl.N, wl.Q, wl.m
    nce = wl.meta["n_ctx_entries"]
    kv = torch.empty((1, N, 512), dtype=torch.bfloat16, device=DEV)
    kv[0, :nce] = wl["kv_ctx"][0]
    pos0 = torch.tensor([wl.meta["pos0"]], dtype=torch.int64, device=DEV)
    buf = P.alloc_prefill(Q, N, 64, 512, DEV, wl.q_pos, m, out_dtype=torch.float32)
    P.prefill_chunk_step(wl["Ca"], wl["Cb"], wl["Za"], wl["Zb"], wl["Ba"], wl["Bb"], wl["prev_Cb"], wl["prev_Zb"],
                         kv, nce, pos0, m, wl["qI"], wl["w"], wl["KI"], wl["q"], wl["swa"], wl.meta["swa_pos0"],
                         wl.q_pos, wl["sink"], buf)
    C.csa2_ctx_check()
    # compressor: the new entries, against the oracle's overlapped compressor
    E = O.compress(_np(wl["Ca"]), _np(wl["Za"]), m, _np(wl["Ba"]), _np(wl["Cb"]), _np(wl["Zb"]), _np(wl["Bb"]),
                   _np(wl["prev_Cb"]), _np(wl["prev_Zb"]))
    new_ref = O.compress_write(E, O.NORM_W | O.ROPE_W, m, wl.meta["pos0"])
    assert_close(to_np(kv[0, nce:].float()), new_ref, 2e-2, "compressed chunk")
    kv_ref = np.concatenate([_np(wl["kv_ctx"][0]), new_ref])
    K_np = _np(wl["KI"][0])
    for qi in (0, 1, 4095, Q - 2, Q - 1):
        t = int(wl.q_pos[0, qi])
        V = t // m
        sc = O.index_score(_np(wl["qI"][0, qi]), _np(wl["w"][0, qi]), K_np, V)
        assert_close(to_np(buf.scores[0, qi]), sc, 1e-5, f"scores q{qi}")
        topk_swaps(to_np(buf.idx[0, qi]), sc, V, 512)
        ref_idx = O.topk(sc, V, 512)
        o, _, _ = O.sparse_attn(_np(wl["q"][0, qi]), kv_ref, ref_idx, _np(wl["swa"][0]), wl.meta["swa_pos0"], t,
                                _np(wl["sink"]), 128)
        g = _gpu_attn_one(wl["q"][0, qi], kv[0], ref_idx, wl["swa"][0], t, wl["sink"], wl.meta["swa_pos0"])
        assert_close(g, o, 2e-2, f"attention q{qi}")


def test_fp4_decode_v4pro_variant():
    """The V4-Pro configuration (DSA-to-CSA/HCA page, «两个已公开配置»): CSA top-1024,
    128 query heads (two 64-head tensor-core passes over the same selected rows),
    64 indexer heads; FP4 caches, 4 sequences of 262,144 entries; sampled sequences
    through the oracle."""
    B, N, H, k = 4, 1 << 18, 128, 1024
    wl = W.fp4_decode(DEV, B=B, N=N, H=H)
    kv = torch.empty((B, N, 288), dtype=torch.uint8, device=DEV)
    ki = torch.empty((B, N, 68), dtype=torch.uint8, device=DEV)
    for b in range(B):
        C.csa2_fp4_pack(W.fp4_rows("kv", b, 0, N, N, DEV), C.FP4_E4M3x16, out=kv[b])
        C.csa2_fp4_pack(W.fp4_rows("KI", b, 0, N, N, DEV), C.MXFP4_E8M0x32, out=ki[b])
    nv = P.visible_entries(wl.q_pos, 1)
    sink = W.normal_tensor((H,), 4109, 0, torch.float32, DEV)
    buf = P.alloc_decode(B, 1, N, H, 512, DEV, out_dtype=torch.float32, k=k)
    P.full_decode_step(wl["qI"], wl["w"], ki, wl["q"], kv, wl["swa"], wl.q_pos, nv, sink, buf, k=k)
    C.csa2_ctx_check()
    t = N - 1
    for b in (0, B - 1):
        ki_ref = O.mxfp4_pack(W.fp4_rows("KI", b, 0, N, N, "cpu").numpy())
        qI_ref = O.mxfp4_pack(wl["qI"][b, 0].float().cpu().numpy())
        V = N - 1
        _, ref_idx = _check_decode_query(b, V, O.mxfp4_unpack(qI_ref), _np(wl["w"][b, 0]),
                                         O.mxfp4_unpack(ki_ref[:V]), to_np(buf.idx[b, 0]), to_np(buf.pool[b, 0]),
                                         to_np(buf.block_max[b, 0]), k=k)
        rows = {int(s): O.nvfp4_unpack(O.nvfp4_pack(W.fp4_rows("kv", b, int(s), 1, N, "cpu").numpy()))[0]
                for s in ref_idx if s >= 0}
        o, _, _ = O.sparse_attn(_np(wl["q"][b, 0]), _RowMap(rows), ref_idx, _np(wl["swa"][b]), 0, t, _np(sink), 128)
        assert o.shape[0] == H
        if np.array_equal(to_np(buf.idx[b, 0]), ref_idx):
            assert_close(to_np(buf.out[b, 0]), o, 2e-2, f"attention (pipeline) b{b}")
        g = _gpu_attn_one(wl["q"][b, 0], kv[b], ref_idx, wl["swa"][b], t, sink)
        assert_close(g, o, 2e-2, f"attention b{b}")


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
        topk_swaps(to_np(idx[b, 0]), ref_sc, V, k)
        ref_idx = O.topk(ref_sc, V, k)
        o, _, _ = O.sparse_attn(_np(q[b, 0]), _np(kv[b]), ref_idx, _np(swa[b]), 0, int(q_pos[b, 0]), _np(sink), 128)
        g = _gpu_attn_one(q[b, 0], kv[b], ref_idx, swa[b], int(q_pos[b, 0]), sink)
        assert_close(g, o, 2e-2, f"attention b{b}")
