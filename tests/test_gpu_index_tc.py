"""GPU parity of the tensor-core indexer scans (64 heads, N a multiple of 8) against
the oracle: full scans with ragged visible counts, several queries sharing a key
tile, pooled candidates, exact-grid inputs (bit-exact) and extreme MXFP4 scales.
Kinds: "bf16" (bf16 q and K), "mx" (bf16 q, MXFP4 K; kind::f16 scan) and "mxq"
(MXFP4 q and K: the FP4 QK path, kind::mxf4), where the oracle scores the
dequantised MXFP4 query."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    yield
    C.csa2_ctx_check()


def _keys(B, N, seed, kind, grid=False, extreme=False):
    KI = W.normal_tensor((B, N, 128), seed, 3, torch.float64, DEV) * torch.exp(
        0.5 * W.normal_tensor((B, N, 1), seed, 4, torch.float64, DEV))
    if extreme:
        # per-32 block scales far apart: 2^-40 .. 2^60 within one row
        e = (W.uniform(B * N * 4, seed, 5, DEV) * 100 - 40).floor().view(B, N, 4, 1)
        KI = (KI.view(B, N, 4, 32) * torch.pow(2.0, e)).view(B, N, 128)
    if grid:
        KI = torch.clamp(torch.round(KI * 2) / 2, -4, 4)
    if kind in ("mx", "mxq"):
        kf = KI.float().reshape(B * N, 128)
        kI = C.csa2_fp4_pack(kf, C.MXFP4_E8M0x32).reshape(B, N, 68)
        K_np = O.mxfp4_unpack(O.mxfp4_pack(kf.cpu().numpy())).reshape(B, N, 128)
    else:
        kI = KI.to(torch.bfloat16)
        K_np = kI.double().cpu().numpy()
    return kI, K_np


def _queries(B, Q, seed, grid=False):
    qI = W.normal_tensor((B, Q, 64, 128), seed, 1, torch.float64, DEV)
    w = W.normal_tensor((B, Q, 64), seed, 2, torch.float64, DEV)
    if grid:
        qI = torch.clamp(torch.round(qI * 8) / 8, -4, 4)
        w = torch.round(w * 2) / 2
    return qI.to(torch.bfloat16), w.float()


def _q_as(kind, qI):
    """(query passed to the scan, its values for the oracle [B, Q, 64, 128] f64)."""
    if kind != "mxq":
        return qI, qI.double().cpu().numpy()
    B, Q = qI.shape[:2]
    qf = qI.float().reshape(-1, 128)
    packed = C.csa2_fp4_pack(qf, C.MXFP4_E8M0x32).reshape(B, Q, 64, 68)
    ref = O.mxfp4_pack(qf.cpu().numpy())
    assert np.array_equal(packed.reshape(-1, 68).cpu().numpy(), ref)
    return packed, O.mxfp4_unpack(ref).reshape(B, Q, 64, 128)


@pytest.mark.parametrize("kind", ["mx", "bf16", "mxq"])
@pytest.mark.parametrize("grid", [False, True])
def test_full_scan_decode(kind, grid):
    B, Q, N = 4, 1, 128 * 37 + 24
    kI, K_np = _keys(B, N, 101, kind, grid)
    qI, w = _queries(B, Q, 102, grid)
    qI, qn = _q_as(kind, qI)
    nv = torch.tensor([[N], [N - 3], [1], [129]], dtype=torch.int64, device=DEV)
    sc, bm = C.csa2_index_score(qI, w, kI, nv, want_block_max=True)
    sc, bm = to_np(sc), to_np(bm)
    for b in range(B):
        V = int(nv[b, 0])
        ref = O.index_score(qn[b, 0], w[b, 0].double().cpu().numpy(), K_np[b], V)
        full_bm = np.full((N + 7) // 8, -np.inf)
        rb = O.block_max(ref, V, 8)
        full_bm[: len(rb)] = rb
        if grid:
            np.testing.assert_array_equal(sc[b, 0], ref)
            np.testing.assert_array_equal(bm[b, 0], full_bm)
        else:
            assert_close(sc[b, 0], ref, 1e-5, f"scores {kind} b{b}")
            assert_close(bm[b, 0], full_bm, 1e-5, f"block max {kind} b{b}")


@pytest.mark.parametrize("kind", ["bf16", "mxq"])
def test_full_scan_several_queries_share_tiles(kind):
    # Q = 10 queries per sequence (bf16: four queries per key tile), causal
    B, Q, N = 2, 10, 128 * 9 + 16
    kI, K_np = _keys(B, N, 111, kind)
    qI, w = _queries(B, Q, 112)
    qI, qn = _q_as(kind, qI)
    nv = torch.tensor([[N, N - 1, N - 2, 900, 800, 128, 127, 1, 0, 555],
                       [5, 500, 1000, N, N, N, 64, 65, 66, 67]], dtype=torch.int64, device=DEV)
    sc, _ = C.csa2_index_score(qI, w, kI, nv)
    sc = to_np(sc)
    for b in range(B):
        for q in range(Q):
            V = int(nv[b, q])
            ref = O.index_score(qn[b, q], w[b, q].double().cpu().numpy(), K_np[b], V)
            assert_close(sc[b, q], ref, 1e-5, f"b{b} q{q}")


@pytest.mark.parametrize("kind", ["mx", "bf16", "mxq"])
def test_candidates_at_the_cache_edges(kind):
    """Pooled blocks at both ends of the key buffer (the first block of the first
    sequence, the last block of the last one: the copies reach the buffer's last row),
    block ids past the cache (skipped: -inf) and -1 padding, on the grid so that the
    scores are bit-exact."""
    B, N, n_pool = 2, 8 * 1024, 64
    kI, K_np = _keys(B, N, 141, kind, grid=True)
    qI, w = _queries(B, 1, 142, grid=True)
    qI, qn = _q_as(kind, qI)
    nv = torch.tensor([[N - 1], [N]], dtype=torch.int64, device=DEV)
    nb = N // 8
    pool = torch.full((B, 1, n_pool), -1, dtype=torch.int32)
    for b in range(B):
        mid = W.distinct_sample(nb - 2, 40, 143, b) + 1
        ids = torch.cat([torch.tensor([0, nb - 1]), mid, torch.tensor([nb, nb + 5])])   # nb, nb + 5: past the cache
        pool[b, 0, :ids.numel()] = torch.sort(ids).values.to(torch.int32)
    pool = pool.to(DEV)
    sc, _ = C.csa2_index_score(qI, w, kI, nv, pool=pool)
    sc = to_np(sc)
    for b in range(B):
        V = int(nv[b, 0])
        full = O.index_score(qn[b, 0], w[b, 0].double().cpu().numpy(), K_np[b], V)
        pl = to_np(pool[b, 0])
        exp = np.full(n_pool * 8, -np.inf)
        for c_ in range(n_pool * 8):
            blk = int(pl[c_ // 8])
            s_ = blk * 8 + c_ % 8
            if 0 <= blk < nb and s_ < V:
                exp[c_] = full[s_]
        assert np.array_equal(sc[b, 0], exp), f"candidates at the edges {kind} b{b}"


@pytest.mark.parametrize("kind", ["mx", "mxq"])
def test_mx_extreme_block_scales(kind):
    B, N = 2, 1024
    kI, K_np = _keys(B, N, 121, kind, extreme=True)
    qI, w = _queries(B, 1, 122)
    qI, qn = _q_as(kind, qI)
    nv = torch.tensor([[N], [N - 100]], dtype=torch.int64, device=DEV)
    sc, _ = C.csa2_index_score(qI, w, kI, nv)
    sc = to_np(sc)
    for b in range(B):
        V = int(nv[b, 0])
        ref = O.index_score(qn[b, 0], w[b, 0].double().cpu().numpy(), K_np[b], V)
        # each score is dominated by its largest block; per-element relative check
        fin = np.isfinite(ref)
        err = np.abs(sc[b, 0][fin] - ref[fin])
        scale = np.abs(ref[fin]) + 1e-30
        bound = 1e-5 * np.maximum(scale, np.abs(O.index_score(np.abs(qn[b, 0]),
                                                              np.abs(w[b, 0].double().cpu().numpy()),
                                                              np.abs(K_np[b]), V))[fin])
        assert np.all(err <= bound), f"worst {np.max(err / bound):.3e}"
        assert np.array_equal(np.isfinite(sc[b, 0]), fin)


@pytest.mark.parametrize("kind", ["mx", "bf16", "mxq"])
@pytest.mark.parametrize("n_pool", [64, 2048])
def test_candidates(kind, n_pool):
    B, N = 3, 8 * 4096
    kI, K_np = _keys(B, N, 131, kind)
    qI, w = _queries(B, 1, 132)
    qI, qn = _q_as(kind, qI)
    nv = torch.tensor([[N - 1], [20001], [333]], dtype=torch.int64, device=DEV)
    pool = torch.full((B, 1, n_pool), -1, dtype=torch.int32)
    for b in range(B):
        V = int(nv[b, 0])
        nb = (V + 7) // 8
        k = min(n_pool - 5, nb - 1)
        sel = W.distinct_sample(nb - 1, k, 133, b)
        pool[b, 0, :k + 1] = torch.sort(torch.cat([sel, torch.tensor([nb - 1])])).values.to(torch.int32)
    pool = pool.to(DEV)
    sc, _ = C.csa2_index_score(qI, w, kI, nv, pool=pool)
    sc = to_np(sc)
    for b in range(B):
        V = int(nv[b, 0])
        full = O.index_score(qn[b, 0], w[b, 0].double().cpu().numpy(), K_np[b], V)
        pl = to_np(pool[b, 0])
        exp = np.full(n_pool * 8, -np.inf)
        for c_ in range(n_pool * 8):
            blk = pl[c_ // 8]
            s = blk * 8 + c_ % 8
            if blk >= 0 and s < V:
                exp[c_] = full[s]
        assert_close(sc[b, 0], exp, 1e-5, f"candidates {kind} b{b}")


@pytest.mark.parametrize("kind", ["mx", "mxq"])
def test_tc_equals_cuda_core_on_grid(kind):
    # the same exact-grid problem through the tensor-core path (N % 8 == 0) and the
    # CUDA-core path (N % 8 != 0, one extra invisible entry): identical scores
    B, N = 2, 128 * 5
    kI, K_np = _keys(B, N + 1, 141, kind, grid=True)
    qI, w = _queries(B, 1, 142, grid=True)
    qI, _ = _q_as(kind, qI)
    nv = torch.tensor([[N], [N - 77]], dtype=torch.int64, device=DEV)
    sc_tc, _ = C.csa2_index_score(qI, w, kI[:, :N].contiguous(), nv)
    sc_cc, _ = C.csa2_index_score(qI, w, kI, nv)
    np.testing.assert_array_equal(to_np(sc_tc), to_np(sc_cc)[:, :, :N])


@pytest.mark.parametrize("kind", ["mx", "mxq"])
def test_bounded_wait_times_out_and_context_recovers(kind):
    """A producer that never signals (test hook): the consumers' bounded waits expire
    (about 2^27 cycles here), the kernel reports a timeout instead of hanging, and
    the next launch on the same context is correct."""
    B, N = 1, 1024
    kI, K_np = _keys(B, N, 151, kind)
    qI, w = _queries(B, 1, 152)
    qI, qn = _q_as(kind, qI)
    nv = torch.tensor([[N]], dtype=torch.int64, device=DEV)
    C.csa2_ctx_test_stall_next(1 << 27)
    C.csa2_index_score(qI, w, kI, nv)
    with pytest.raises(C.Csa2Error) as e:
        C.csa2_ctx_check()
    assert e.value.status == C.ERR_TIMEOUT
    sc, _ = C.csa2_index_score(qI, w, kI, nv)
    C.csa2_ctx_check()
    ref = O.index_score(qn[0, 0], w[0, 0].double().cpu().numpy(), K_np[0], N)
    assert_close(to_np(sc)[0, 0], ref, 1e-5, "after timeout")


@pytest.mark.parametrize("B,Q,N", [(1, 1, 8), (2, 3, 4096), (8, 1, 131072)])
def test_in_scan_query_packing_equals_separate_pack(B, Q, N):
    """csa2_index_score_mxq (the bf16 query packed to MXFP4 inside the FP4 scan) gives
    the bytes of csa2_fp4_pack and then the same scores, block maxima and histogram as
    csa2_index_score on that packed query, bit for bit; the scores match the oracle on
    the dequantised packed query.  Visible counts ragged, some 0, some past N."""
    kI, K_np = _keys(B, N, 171 + N, "mx")
    qI, w = _queries(B, Q, 172 + N)
    vis = [(N * (3 * i + 1)) // (3 * B * Q) for i in range(B * Q)]
    vis[0] = 0 if B * Q > 1 else N
    vis[-1] = N + 5
    nv = torch.tensor(vis, dtype=torch.int64, device=DEV).view(B, Q)
    nb = N // 8
    packed = torch.empty((B, Q, 64, 68), dtype=torch.uint8, device=DEV)
    sc1, bm1 = C.csa2_index_score_mxq(qI, w, kI, nv, want_block_max=True, q_mx_out=packed,
                                      block_hist=torch.empty((B, Q, C.BLOCK_HIST_BINS), dtype=torch.int32, device=DEV))
    qmx = C.csa2_fp4_pack(qI, C.MXFP4_E8M0x32)
    hist2 = torch.empty((B, Q, C.BLOCK_HIST_BINS), dtype=torch.int32, device=DEV)
    sc2, bm2 = C.csa2_index_score(qmx, w, kI, nv, want_block_max=True, block_hist=hist2)
    # the histogram of the first call, read back through a second call into its own buffer
    hist1 = torch.empty_like(hist2)
    C.csa2_index_score_mxq(qI, w, kI, nv, want_block_max=True, block_hist=hist1)
    C.csa2_ctx_check()
    assert torch.equal(packed, qmx)
    assert torch.equal(sc1, sc2) and torch.equal(bm1, bm2) and torch.equal(hist1, hist2)
    q_np = O.mxfp4_unpack(qmx.reshape(-1, 68).cpu().numpy()).reshape(B, Q, 64, 128)
    for b, q in [(0, 0), (B - 1, Q - 1)]:
        V = min(int(nv[b, q]), N)
        ref = O.index_score(q_np[b, q], w[b, q].double().cpu().numpy(), K_np[b], V)
        assert_close(to_np(sc1[b, q]), ref, 1e-5, f"b{b} q{q}")
