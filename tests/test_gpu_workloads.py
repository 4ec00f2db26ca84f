"""Whole-path parity on the five workloads, at their full sizes and in the launch
configuration bench.py times, checked against the oracle on sampled sequences /
queries (the oracle computes those one by one)."""
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
    out, _ = C.csa2_sparse_attn(wl["q"], kv.unsqueeze(0), idx, wl["swa"], wl.q_pos, wl["sink"], window=128,
                                want_lse=False)
    for qi, t in enumerate(wl.q_pos[0].tolist()):
        V = t // 2
        ref_sc = O.index_score(_np(wl["qI"][0, qi]), _np(wl["w"][0, qi]), _np(wl["KI"][0]), V)
        assert_close(to_np(sc)[0, qi], ref_sc, 1e-4, f"scores q{qi}")
        topk_swaps(to_np(idx)[0, qi], ref_sc, V, 512)
        # attention given the same indices, against the oracle's own compressed cache
        o, _, _ = O.sparse_attn(_np(wl["q"][0, qi]), kv_ref, to_np(idx)[0, qi], _np(wl["swa"][0]), 0, t,
                                _np(wl["sink"]), 128)
        assert_close(to_np(out)[0, qi], o, 1e-4, f"attention q{qi}")


def _check_decode_query(b, V, qI, w, K_np, gpu_idx, gpu_pool, gpu_bmax, k=512, n_keep=2048):
    sc = O.index_score(qI, w, K_np, V)
    swaps = topk_swaps(gpu_idx, sc, V, k)
    if gpu_bmax is not None:
        bm = O.block_max(sc, V, 8)
        assert_close(gpu_bmax[: len(bm)], bm, 1e-5, f"block max b{b}")
    if gpu_pool is not None:
        pool_swaps(gpu_pool, O.block_max(sc, V, 8), V, 8, n_keep)
        # the top-k lies inside the pool
        cand = set(O.pool_candidates(gpu_pool, V).tolist())
        assert set(int(i) for i in gpu_idx if i >= 0) <= cand
    return sc, swaps


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
        sc, swaps = _check_decode_query(b, V, _np(wl["qI"][b, 0]), _np(wl["w"][b, 0]), K_np,
                                        to_np(buf.idx[b, 0]), to_np(buf.pool[b, 0]), to_np(buf.block_max[b, 0]))
        idx = to_np(buf.idx[b, 0])
        rows = {int(s): O.nvfp4_unpack(O.nvfp4_pack(W.fp4_rows("kv", b, int(s), 1, N, "cpu").numpy()))[0]
                for s in idx if s >= 0}
        o, _, _ = O.sparse_attn(_np(wl["q"][b, 0]), _RowMap(rows), idx, _np(wl["swa"][b]), 0, t,
                                _np(wl["sink"]), 128)
        assert_close(to_np(buf.out[b, 0]), o, 2e-2, f"attention b{b}")
        # the new token's main-KV row: RoPE'd copy of C_new (m = 1), FP4-packed
        new_ref = O.compress_write(_np(wl["C_new"][b]), O.ROPE_W, 1, t)
        got = O.nvfp4_unpack(to_np(kv[b, t:t + 1]))[0]
        ref = O.nvfp4_unpack(O.nvfp4_pack(new_ref.astype(np.float32)))[0]
        s = np.repeat(O.e4m3_decode(to_np(kv[b, t, 256:])), 16)
        assert np.all(np.abs(got - ref) <= 2 * s + 1e-6)


class _RowMap:
    def __init__(self, rows):
        self.rows = rows

    def __getitem__(self, s):
        return self.rows[int(s)]


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
        sc, _ = _check_decode_query(b, V, _np(wl["qI"][b, 0]), _np(wl["w"][b, 0]), _np(wl["KI"][b]),
                                    to_np(buf.idx[b, 0]), to_np(buf.pool[b, 0]), to_np(buf.block_max[b, 0]))
        planted = to_np(wl["planted"][b])
        mu, sd = sc[:4096].mean(), sc[:4096].std()
        assert np.all(sc[planted] >= mu + 8 * sd)
        assert set(planted.tolist()) <= set(to_np(buf.idx[b, 0]).tolist())
        assert set((planted // 8).tolist()) <= set(to_np(buf.pool[b, 0]).tolist())
        rows = {int(s): _np(wl["kv"][b, int(s)]) for s in to_np(buf.idx[b, 0]) if s >= 0}
        o, _, _ = O.sparse_attn(_np(wl["q"][b, 0]), _RowMap(rows), to_np(buf.idx[b, 0]), _np(wl["swa"][b]), 0, t,
                                _np(wl["sink"]), 128)
        assert_close(to_np(buf.out[b, 0]), o, 2e-2, f"attention b{b}")


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
        rows = {int(s): _np(wl["kv"][b, int(s)]) for s in gpu if s >= 0}
        for l in range(4):
            o, _, _ = O.sparse_attn(_np(wl[f"q{l}"][b, 0]), _RowMap(rows), gpu, _np(wl[f"swa{l}"][b]), 0, t,
                                    _np(wl["sink"]), 128)
            assert_close(to_np(outs[l][b, 0].float()), o, 2e-2, f"layer {l} b{b}")
