"""GPU parity of each C-ABI entry point against the oracle (seeded inputs, sizes
that span several tiles and a ragged tail, plus the edge cases)."""
import math

import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np, topk_swaps

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    yield
    C.csa2_ctx_check()


def _rows(n, width, seed, dtype):
    x = W.normal_tensor((n, width), seed, 0, torch.float64, DEV)
    r = torch.exp(0.5 * W.normal_tensor((n, 1), seed, 1, torch.float64, DEV))
    return (x * r).to(dtype)


def _edge_rows(width, dtype):
    """Rows that hit the format's corner cases."""
    rows = []
    z = torch.zeros(width, dtype=torch.float64)
    rows.append(z.clone())                                      # all zero
    r = z.clone(); r[: width // 2] = -0.0; rows.append(r)       # negative zeros
    r = torch.full((width,), 1e-5, dtype=torch.float64); r[1::2] *= -1; rows.append(r)   # tiny
    r = torch.full((width,), 1e4, dtype=torch.float64); r[::3] *= -0.37; rows.append(r)  # huge
    ties = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5,
                         -5.0, -6.0], dtype=torch.float64)
    rows.append(ties.repeat(width // 16))                       # RNE ties at scale 1
    r = torch.linspace(-7, 7, width, dtype=torch.float64); rows.append(r)
    r = torch.full((width,), 2.0 ** -130, dtype=torch.float64); r[0] = 2.0 ** -128; rows.append(r)  # subnormal
    r = torch.full((width,), 448.0 * 6, dtype=torch.float64); rows.append(r)             # scale at E4M3 max
    return torch.stack(rows).to(dtype).to(DEV)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [C.FP4_E4M3x16, C.MXFP4_E8M0x32])
def test_fp4_pack_unpack_bit_exact(dtype, fmt):
    width = 512 if fmt == C.FP4_E4M3x16 else 128
    x = torch.cat([_rows(3001, width, 77, dtype), _edge_rows(width, dtype)])
    got = to_np(C.csa2_fp4_pack(x, fmt))
    xo = x.float().cpu().numpy()
    ref = O.nvfp4_pack(xo) if fmt == C.FP4_E4M3x16 else O.mxfp4_pack(xo)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:5].tolist()}"
    b = torch.from_numpy(ref).to(DEV)
    for odt in (torch.float32, torch.bfloat16):
        un = to_np(C.csa2_fp4_unpack(b, fmt, width, odt))
        exp = O.nvfp4_unpack(ref, width) if fmt == C.FP4_E4M3x16 else O.mxfp4_unpack(ref, width)
        np.testing.assert_array_equal(un, exp)


@pytest.mark.parametrize("case", ["nonoverlap_f32_m2", "overlap_bf16_m4_state", "overlap_f32_m4_nostate",
                                  "m1_identity_rope"])
def test_compress(case):
    c = 512
    if case == "nonoverlap_f32_m2":
        m, n, dt, overlap, state, flags = 2, 2 * 301, torch.float32, False, False, C.W_NORM | C.W_ROPE
    elif case == "overlap_bf16_m4_state":
        m, n, dt, overlap, state, flags = 4, 4 * 203, torch.bfloat16, True, True, C.W_NORM | C.W_ROPE
    elif case == "overlap_f32_m4_nostate":
        m, n, dt, overlap, state, flags = 4, 4 * 77, torch.float32, True, False, 0
    else:
        m, n, dt, overlap, state, flags = 1, 37, torch.bfloat16, False, False, C.W_ROPE
    g = lambda s, shape, std=1.0: W.normal_tensor(shape, 900 + s, 0, dt if s < 6 else torch.float32, DEV, std=std)
    Ca, Za, Cb, Zb = g(1, (n, c)), g(2, (n, c)), g(3, (n, c)), g(4, (n, c))
    Ba, Bb = g(6, (m, c), 0.1), g(7, (m, c), 0.1)
    pCb, pZb = g(8, (m, c)).to(dt), g(9, (m, c)).to(dt)
    pos0 = 131072
    kw = dict(ba=Ba, pos0=pos0, flags=flags)
    if overlap:
        kw.update(cb=Cb, zb=Zb, bb=Bb)
        if state:
            kw.update(prev_cb=pCb, prev_zb=pZb)
    out = C.csa2_compress(Ca, Za, m, out_fmt="f32" if dt == torch.float32 else "bf16", **kw)
    npy = lambda t: None if t is None else t.double().cpu().numpy()
    E = O.compress(npy(Ca), npy(Za), m, npy(Ba), npy(Cb) if overlap else None, npy(Zb) if overlap else None,
                   npy(Bb) if overlap else None, npy(pCb) if state else None, npy(pZb) if state else None)
    ref = O.compress_write(E, flags, m, pos0)
    assert_close(to_np(out), ref, 1e-4 if dt == torch.float32 else 2e-2, case)
    if m == 1 and flags == C.W_ROPE:
        # m = 1: the entry is its token, only rotated
        np.testing.assert_allclose(to_np(out)[:, :448], npy(Ca)[:, :448], rtol=0, atol=0)
    # the fused FP4 store equals packing the f32 result with csa2_fp4_pack
    out32 = C.csa2_compress(Ca, Za, m, out_fmt="f32", **kw)
    packed = C.csa2_compress(Ca, Za, m, out_fmt="fp4", **kw)
    np.testing.assert_array_equal(to_np(packed), to_np(C.csa2_fp4_pack(out32)))


def test_compress_worked_example_padded():
    # The pages' csa_compress example (m=2, c=3) embedded in 128 channels.
    g = O  # noqa: F841
    Ca = torch.zeros((4, 128), device=DEV)
    Cb = torch.zeros((4, 128), device=DEV)
    Ca[:2, :3], Ca[2:, :3] = 1.0, 3.0
    Cb[:2, :3], Cb[2:, :3] = 2.0, 4.0
    Z = torch.zeros_like(Ca)
    y = to_np(C.csa2_compress(Ca, Z, 2, cb=Cb, zb=Z))
    np.testing.assert_array_equal(y[0, :3], [1, 1, 1])
    np.testing.assert_array_equal(y[1, :3], [2.5, 2.5, 2.5])


def _index_inputs(B, Q, N, H_I, seed, q_dt, k_kind, grid=False):
    qI = W.normal_tensor((B, Q, H_I, 128), seed, 1, torch.float64, DEV)
    w = W.normal_tensor((B, Q, H_I), seed, 2, torch.float64, DEV)
    KI = W.normal_tensor((B, N, 128), seed, 3, torch.float64, DEV) * torch.exp(
        0.5 * W.normal_tensor((B, N, 1), seed, 4, torch.float64, DEV))
    if grid:
        # exact-grid inputs: every partial sum is exact in f32 in any order
        qI = torch.clamp(torch.round(qI * 8) / 8, -4, 4)
        KI = torch.clamp(torch.round(KI * 2) / 2, -4, 4)
        w = torch.round(w * 2) / 2
    w = w.float()
    if q_dt == "mx":
        # MXFP4 queries (the FP4 QK path); the oracle scores their dequantised values
        qf = qI.float().reshape(-1, 128)
        qI = C.csa2_fp4_pack(qf, C.MXFP4_E8M0x32).reshape(B, Q, H_I, 68)
        q_ref = O.mxfp4_pack(qf.cpu().numpy())
        assert np.array_equal(qI.reshape(-1, 68).cpu().numpy(), q_ref)
        qn = O.mxfp4_unpack(q_ref).reshape(B, Q, H_I, 128)
    else:
        qI = qI.to(q_dt)
        qn = qI.double().cpu().numpy()
    if k_kind == "mx":
        kI = C.csa2_fp4_pack(KI.float().reshape(B * N, 128), C.MXFP4_E8M0x32).reshape(B, N, 68)
        K_np = O.mxfp4_unpack(O.mxfp4_pack(KI.float().reshape(B * N, 128).cpu().numpy())).reshape(B, N, 128)
    else:
        kI = KI.to(torch.float32 if k_kind == "f32" else torch.bfloat16)
        K_np = kI.double().cpu().numpy()
    return qI, w, kI, K_np, qn


@pytest.mark.parametrize("q_dt,k_kind,H_I", [(torch.float32, "f32", 8), (torch.bfloat16, "bf16", 64),
                                             (torch.bfloat16, "mx", 64), (torch.float32, "mx", 8),
                                             ("mx", "mx", 64), ("mx", "mx", 8), ("mx", "bf16", 8)])
@pytest.mark.parametrize("grid", [False, True])
def test_index_score_full_scan(q_dt, k_kind, H_I, grid):
    """N = 1357 (ten tiles and a ragged one; N % 8 != 0 takes the CUDA-core path, so
    the 64-head MXFP4 cases also run N = 1352 on the tensor cores)."""
    for N in ((1000 + 357, 1000 + 352) if H_I == 64 else (1000 + 357,)):
        _full_scan_case(q_dt, k_kind, H_I, grid, N)


def _full_scan_case(q_dt, k_kind, H_I, grid, N):
    B, Q = 2, 3
    qI, w, kI, K_np, qn = _index_inputs(B, Q, N, H_I, 31, q_dt, k_kind, grid)
    nv = torch.tensor([[N, N - 1, 0], [777, 1, N - 8]], dtype=torch.int64, device=DEV)
    sc, bm = C.csa2_index_score(qI, w, kI, nv, want_block_max=True)
    sc, bm = to_np(sc), to_np(bm)
    wn = w.double().cpu().numpy()
    for b in range(B):
        for q in range(Q):
            V = int(nv[b, q])
            ref = O.index_score(qn[b, q], wn[b, q], K_np[b], V)
            if grid:
                np.testing.assert_array_equal(sc[b, q], ref)        # exact in f32 in any order
            else:
                assert_close(sc[b, q], ref, 1e-4, f"scores b{b} q{q}")
            refb = O.block_max(ref, V, 8)
            nb = (N + 7) // 8
            full = np.full(nb, -np.inf)
            full[: len(refb)] = refb
            if grid:
                np.testing.assert_array_equal(bm[b, q], full)
            else:
                assert_close(bm[b, q], full, 1e-4, "block max")


@pytest.mark.parametrize("q_dt,k_kind", [(torch.bfloat16, "bf16"), (torch.bfloat16, "mx"), ("mx", "mx")])
def test_index_score_candidates(q_dt, k_kind):
    B, Q, N, H_I = 2, 1, 5000, 64
    qI, w, kI, K_np, qn = _index_inputs(B, Q, N, H_I, 41, q_dt, k_kind)
    nv = torch.tensor([[N - 3], [4000]], dtype=torch.int64, device=DEV)
    n_pool = 300
    pool = torch.full((B, Q, n_pool), -1, dtype=torch.int32)
    for b in range(B):
        V = int(nv[b, 0])
        nb = (V + 7) // 8
        sel = W.distinct_sample(nb - 1, 250, 55, b)
        pool[b, 0, :251] = torch.sort(torch.cat([sel, torch.tensor([nb - 1])])).values.to(torch.int32)
    pool = pool.to(DEV)
    sc, _ = C.csa2_index_score(qI, w, kI, nv, pool=pool)
    idx, val = C.csa2_topk(sc, nv, 512, pool=pool, want_scores=True)
    sc, idx = to_np(sc), to_np(idx)
    wn = w.double().cpu().numpy()
    for b in range(B):
        V = int(nv[b, 0])
        full = O.index_score(qn[b, 0], wn[b, 0], K_np[b], V)
        pl = to_np(pool[b, 0])
        for c_ in range(n_pool * 8):
            blk = pl[c_ // 8]
            s = blk * 8 + c_ % 8
            if blk < 0 or s >= V:
                assert sc[b, 0, c_] == -np.inf
            else:
                assert abs(sc[b, 0, c_] - full[s]) <= 1e-4 * (abs(full[s]) + 64)
        ref = O.reindex_topk(full, pl, V, 512)
        cand = O.pool_candidates(pl, V)
        masked = np.full(N, -np.inf)
        masked[cand] = full[cand]
        # compare as a top-k restricted to the candidates
        gpu = [i for i in idx[b, 0] if i >= 0]
        assert len(gpu) == len([i for i in ref if i >= 0])
        assert set(gpu) <= set(cand.tolist())
        if gpu != [i for i in ref if i >= 0]:
            kth = np.sort(full[cand])[::-1][511]
            for i in set(gpu) ^ set(int(x) for x in ref if x >= 0):
                assert abs(full[i] - kth) <= 1e-5 * np.sqrt(np.mean(full[:V] ** 2))


def _score_rows(rows, n, seed, ties):
    x = W.normal_tensor((rows, n), seed, 0, torch.float64, DEV)
    if ties:
        x = torch.round(x * 2)           # heavy ties
    x = x.float()
    x[0, ::3] = -0.0                      # negative zeros mixed with zeros
    x[0, 1::3] = 0.0
    return x


@pytest.mark.parametrize("n,k", [(1, 1), (100, 512), (5000, 512), (70001, 512), (16384, 512), (3000, 2048)])
@pytest.mark.parametrize("ties", [False, True])
def test_topk_bit_exact(n, k, ties):
    rows = 5
    s = _score_rows(rows, n, 61 + n, ties)
    nv = torch.tensor([n, max(n - 1, 0), min(n, k), 0, n // 2], dtype=torch.int64, device=DEV)
    idx, val = C.csa2_topk(s, nv, k, want_scores=True)
    idx, val, sn = to_np(idx), to_np(val), s.double().cpu().numpy()
    for r in range(rows):
        ref = O.topk(sn[r], int(nv[r]), k)
        np.testing.assert_array_equal(idx[r], ref)
        exp_val = np.where(ref >= 0, sn[r][np.maximum(ref, 0)], -np.inf)
        np.testing.assert_array_equal(val[r], exp_val)


@pytest.mark.parametrize("n,k,ties", [(5000, 512, False), (5000, 512, True), (40960, 512, False), (2000, 64, True)])
def test_topk_many_rows_bit_exact(n, k, ties):
    """Enough rows (as in prefill) for the one-CTA-per-row streaming kernel; visible
    counts cover full, partial, ragged and empty rows; all rows against the oracle."""
    rows = 400
    s = _score_rows(rows, n, 71 + n, ties)
    nv = torch.tensor([(n - (37 * r) % (n + 1)) if r % 7 else (r % 3) * (k // 2) for r in range(rows)],
                      dtype=torch.int64, device=DEV)
    idx, val = C.csa2_topk(s, nv, k, want_scores=True)
    idx, val, sn = to_np(idx), to_np(val), s.double().cpu().numpy()
    for r in range(rows):
        ref = O.topk(sn[r], int(nv[r]), k)
        np.testing.assert_array_equal(idx[r], ref, err_msg=f"row {r}")
        exp_val = np.where(ref >= 0, sn[r][np.maximum(ref, 0)], -np.inf)
        np.testing.assert_array_equal(val[r], exp_val)


def test_topk_all_equal_scores():
    s = torch.full((2, 10000), 3.25, device=DEV)
    nv = torch.tensor([10000, 600], dtype=torch.int64, device=DEV)
    idx, _ = C.csa2_topk(s, nv, 512)
    np.testing.assert_array_equal(to_np(idx), np.stack([np.arange(512), np.arange(512)]))


@pytest.mark.parametrize("V", [0, 1, 8, 9, 100, 4097, 8 * 2048, 8 * 2048 + 1, 131071, 1048575])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("path", ["histogram", "general"])
def test_block_pool_bit_exact(V, ties, path):
    """Both pool selections: from the row histograms (built in the workspace here; the
    decode step takes them from the scan) with the n_top best blocks as well, and the
    general radix select (a workspace too small for the histograms).  With ties the
    threshold bin is crowded, which takes the histogram path's cluster-wide passes."""
    nb_max = (1048575 + 7) // 8
    n_keep, n_top = 2048, 512
    bm = _score_rows(2, nb_max, 71, ties)
    nv = torch.tensor([V, max(V - 5, 0)], dtype=torch.int64, device=DEV)
    bmn = bm.double().cpu().numpy()
    if path == "histogram":
        pool, top = C.csa2_block_pool(bm, nv, 8, n_keep, n_top=n_top)
        pool, top = to_np(pool), to_np(top)
    else:
        pool = to_np(C.csa2_block_pool(bm, nv, 8, n_keep, ws=torch.empty(16, dtype=torch.uint8, device=DEV)))
    for r in range(2):
        Vr = int(nv[r])
        nb = (Vr + 7) // 8
        ref = O.block_pool(bmn[r][:nb], Vr, 8, n_keep)
        np.testing.assert_array_equal(pool[r], ref)
        if path == "histogram":
            # the n_top best blocks: top-k over the block maxima as scores
            np.testing.assert_array_equal(top[r], O.topk(bmn[r][:nb], nb, n_top))
            assert set(top[r][top[r] >= 0].tolist()) <= set(ref[ref >= 0].tolist())


def test_block_hist_from_scan_equals_from_maxima():
    """The FP4 scan's own histogram of the block maxima drives the same selections as
    the histogram built from the written maxima (the selections themselves are held to
    the oracle by test_block_pool_bit_exact and the full-size workload tests)."""
    B, N = 2, 1 << 18
    ki = torch.stack([C.csa2_fp4_pack(W.fp4_rows("KI", b, 0, N, N, DEV), C.MXFP4_E8M0x32) for b in range(B)])
    qI = C.csa2_fp4_pack(W.normal_tensor((B, 1, 64, 128), 4301, 0, torch.float32, DEV), C.MXFP4_E8M0x32)
    w = W.normal_tensor((B, 1, 64), 4302, 0, torch.float32, DEV)
    nv = torch.tensor([[N - 1], [N - 70000]], dtype=torch.int64, device=DEV)
    hist = torch.empty((B, 1, C.BLOCK_HIST_BINS), dtype=torch.int32, device=DEV)
    _, bm = C.csa2_index_score(qI, w, ki, nv, want_scores=False, want_block_max=True, block_hist=hist)
    p1, t1 = C.csa2_block_pool(bm, nv, 8, 2048, block_hist=hist, n_top=512)
    p2, t2 = C.csa2_block_pool(bm, nv, 8, 2048, n_top=512)
    C.csa2_ctx_check()
    np.testing.assert_array_equal(to_np(p1), to_np(p2))
    np.testing.assert_array_equal(to_np(t1), to_np(t2))


def test_sink_and_worked_example_through_abi(golden):
    """The pages' sparse_shared_kv example through csa2_index_score, csa2_topk and
    csa2_sparse_attn (flags off, no window).  Vectors are zero-padded to the
    library's widths and the query is scaled by sqrt(512/2) so the 1/sqrt(c)
    logit scale equals the example's 1/sqrt(2)."""
    g = golden("sparse_shared_kv_example.json")
    hd = g["hand_derived"]
    iq = torch.zeros((1, 1, 2, 128), device=DEV)
    iq[0, 0, :, :2] = torch.tensor(g["iq"])
    ik = torch.zeros((1, 3, 128), device=DEV)
    ik[0, :, :2] = torch.tensor(g["ik"])
    w = torch.tensor([[g["head_weight"]]], device=DEV)
    nv = torch.tensor([[3]], dtype=torch.int64, device=DEV)
    sc, _ = C.csa2_index_score(iq, w, ik, nv)
    np.testing.assert_array_equal(to_np(sc)[0, 0], hd["scores"])
    idx, _ = C.csa2_topk(sc, nv, g["k"])
    np.testing.assert_array_equal(to_np(idx)[0, 0], hd["ids_ascending"])
    q = torch.zeros((1, 1, 1, 512), device=DEV)
    q[0, 0, 0, :2] = torch.tensor(g["q"]) * math.sqrt(512 / 2)
    kv = torch.zeros((1, 3, 512), device=DEV)
    kv[0, :, :2] = torch.tensor(g["kv"])
    pos = torch.tensor([[0]], dtype=torch.int64, device=DEV)
    sink = torch.tensor([g["sink_logit"]], device=DEV)
    out, lse = C.csa2_sparse_attn(q, kv, idx, None, pos, sink, window=0, flags=0, want_lse=True)
    o = to_np(out)[0, 0, 0]
    np.testing.assert_allclose(o[:2], hd["out"], rtol=1e-6)
    assert np.all(o[2:] == 0)
    a, b = math.exp(math.sqrt(2)), math.exp(1 / math.sqrt(2))
    np.testing.assert_allclose(to_np(lse)[0, 0, 0], math.log(a + b + 1), rtol=1e-6)


@pytest.mark.parametrize("kv_kind", ["f32", "bf16", "fp4"])
@pytest.mark.parametrize("flags", [C.ATTN_DEFAULT, 0, C.QNORM | C.KVNORM])
def test_sparse_attn(kv_kind, flags):
    B, Q, H, N = 2, 3, 16, 3000
    q_dt = torch.float32 if kv_kind == "f32" else torch.bfloat16
    q = W.normal_tensor((B, Q, H, 512), 81, 1, q_dt, DEV)
    kv_f = W.normal_tensor((B, N, 512), 81, 2, torch.float32, DEV) * 1.5
    if kv_kind == "fp4":
        kv = C.csa2_fp4_pack(kv_f)
        kv_np = O.nvfp4_unpack(O.nvfp4_pack(kv_f.reshape(-1, 512).cpu().numpy())).reshape(B, N, 512)
    else:
        kv = kv_f.to(q_dt)
        kv_np = kv.double().cpu().numpy()
    cap = 128
    swa = W.normal_tensor((B, cap, 512), 81, 3, q_dt, DEV)
    q_pos = torch.tensor([[N, 5, 1000], [70, N + 200, 0]], dtype=torch.int64, device=DEV)
    k = 512
    idx = torch.full((B, Q, k), -1, dtype=torch.int32)
    for b in range(B):
        for qq in range(Q):
            V = min(int(q_pos[b, qq]), N)
            n = min(V, [512, 300, 17][qq % 3])
            if n:
                idx[b, qq, :n] = W.distinct_sample(V, n, 83 + b, qq).to(torch.int32)
    idx = idx.to(DEV)
    sink = W.normal_tensor((H,), 81, 4, torch.float32, DEV)
    out, lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=128, flags=flags, out_dtype=torch.float32,
                                  want_lse=True)
    out, lse = to_np(out), to_np(lse)
    tol = 1e-4 if kv_kind == "f32" else 2e-2
    # The tensor-core path (bf16 query, both norms) rounds the normalised query to
    # bf16: a logit q^.k^/sqrt(c) moves by about 2^-9 |q^||k^| / (sqrt(3) c) ~ 1e-3,
    # and lse by the softmax-weighted mean of those moves, up to that size when few
    # keys carry the mass; fp32 paths stay at 1e-5.
    tc = kv_kind != "f32" and (flags & C.QNORM) and (flags & C.KVNORM)
    lse_tol = 2e-3 if tc else 1e-5
    for b in range(B):
        for qq in range(Q):
            t = int(q_pos[b, qq])
            o, l, mass = O.sparse_attn(q[b, qq].double().cpu().numpy(), kv_np[b], to_np(idx[b, qq]),
                                       swa[b].double().cpu().numpy(), 0, t, sink.double().cpu().numpy(), 128, flags)
            assert_close(out[b, qq], o, tol, f"out b{b} q{qq}")
            assert_close(lse[b, qq], l, lse_tol, "lse")
            assert np.all((mass > 0) & (mass < 1))


def test_sparse_attn_linear_window_and_no_sink():
    B, Q, H, N = 1, 2, 8, 500
    q = W.normal_tensor((B, Q, H, 512), 91, 1, torch.bfloat16, DEV)
    kv = W.normal_tensor((B, N, 512), 91, 2, torch.bfloat16, DEV)
    pos0 = 10000
    swa = W.normal_tensor((B, 400, 512), 91, 3, torch.bfloat16, DEV)   # positions 10000..10399
    q_pos = torch.tensor([[10127, 10399]], dtype=torch.int64, device=DEV)
    idx = torch.arange(0, 512, dtype=torch.int32, device=DEV).clamp(max=N - 1).reshape(1, 1, 512).repeat(1, 2, 1)
    idx[:, :, N:] = -1
    out, _ = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, None, window=128, swa_pos0=pos0, out_dtype=torch.float32)
    for qq in range(Q):
        o, _, mass = O.sparse_attn(q[0, qq].double().cpu().numpy(), kv[0].double().cpu().numpy(),
                                   to_np(idx[0, qq]), swa[0].double().cpu().numpy(), pos0, int(q_pos[0, qq]),
                                   None, 128)
        assert_close(to_np(out)[0, qq], o, 2e-2, "linear window")
        np.testing.assert_allclose(mass, 1.0, rtol=1e-12)


def test_out_of_range_index_is_flagged_not_faulted():
    B, Q, H, N = 1, 1, 8, 100
    q = torch.randn((B, Q, H, 512), device=DEV)
    kv = torch.randn((B, N, 512), device=DEV)
    idx = torch.tensor([[[3, 7, N + 5, -1]]], dtype=torch.int32, device=DEV)
    pos = torch.tensor([[50]], dtype=torch.int64, device=DEV)
    C.csa2_sparse_attn(q, kv, idx, None, pos, None, window=0)
    with pytest.raises(C.Csa2Error) as e:
        C.csa2_ctx_check()
    assert e.value.status == C.ERR_DEVICE
    C.csa2_ctx_check()   # cleared


@pytest.mark.parametrize("ties", [False, True])
def test_selection_without_workspace_matches(ties):
    """Rows too long for the cluster path (more than 16 x 16,384 elements) with no
    workspace take the one-CTA-per-row path through global memory; with a
    workspace, the chunk + merge path; the result is the same exact selection."""
    tiny = torch.empty(16, dtype=torch.uint8, device=DEV)
    nbl = 300000
    bm = _score_rows(2, nbl, 171, ties)
    nv = torch.tensor([8 * nbl - 3, 700001], dtype=torch.int64, device=DEV)
    bmn = bm.double().cpu().numpy()
    for ws in (tiny, None):
        pool = to_np(C.csa2_block_pool(bm, nv, 8, 2048, ws=ws))
        for r in range(2):
            Vr = int(nv[r])
            np.testing.assert_array_equal(pool[r], O.block_pool(bmn[r][: (Vr + 7) // 8], Vr, 8, 2048))
    s = _score_rows(3, nbl, 172, ties)
    nv = torch.tensor([nbl, 45000, 100], dtype=torch.int64, device=DEV)
    sn = s.double().cpu().numpy()
    for ws in (tiny, None):
        idx, _ = C.csa2_topk(s, nv, 512, ws=ws)
        for r in range(3):
            np.testing.assert_array_equal(to_np(idx)[r], O.topk(sn[r], int(nv[r]), 512))


@pytest.mark.parametrize("rows,n,k", [(12, 20000, 512), (9, 131072, 2047), (3, 4096, 4096), (19, 9000, 100),
                                      (3, 200000, 512)])
@pytest.mark.parametrize("ties", [False, True])
def test_topk_cluster_rows_bit_exact(rows, n, k, ties):
    """Few long rows: one thread-block cluster per row (8 CTAs; 16 when a row needs more
    than 8 x 16,384 keys, here 200,000).  Visible counts cover full, ragged, tiny, empty
    and <= k rows."""
    s = _score_rows(rows, n, 181 + n + rows, ties)
    nv = torch.tensor([[n, n - 1, 1, 0, k, k + 1, n // 3][r % 7] for r in range(rows)], dtype=torch.int64,
                      device=DEV)
    idx, val = C.csa2_topk(s, nv, k, want_scores=True)
    idx, val, sn = to_np(idx), to_np(val), s.double().cpu().numpy()
    for r in range(rows):
        ref = O.topk(sn[r], int(nv[r]), k)
        np.testing.assert_array_equal(idx[r], ref, err_msg=f"row {r}")
        exp_val = np.where(ref >= 0, sn[r][np.maximum(ref, 0)], -np.inf)
        np.testing.assert_array_equal(val[r], exp_val)


@pytest.mark.parametrize("ties", [False, True])
def test_topk_candidates_cluster_bit_exact(ties):
    """Top-512 over 2,048 pooled blocks x 8 candidates (the decode Reindex shape) on
    the cluster path: empty slots (-1), blocks past the visible count, a partial last
    block; compared with the oracle's restricted top-k."""
    rows, n_pool, N = 6, 2048, 1 << 20
    s = _score_rows(rows, n_pool * 8, 191, ties)
    pool = torch.full((rows, n_pool), -1, dtype=torch.int32)
    nv = [N - 1, 20000, 16383, 333, 9, 0]
    for r in range(rows):
        nb = (nv[r] + 7) // 8
        if nb == 0:
            continue
        m = min(n_pool - 100 * (r % 2) - (r == 0), nb)
        sel = W.distinct_sample(max(nb - 1, 1), m - 1, 193, r) if m > 1 else torch.empty(0, dtype=torch.int64)
        blocks = torch.sort(torch.cat([sel, torch.tensor([nb - 1])])).values
        pool[r, : len(blocks)] = blocks.to(torch.int32)
        if r == 0:
            pool[r, len(blocks)] = nb + 3          # a block past the visible count (pool stays ascending)
    pool = pool.to(DEV)
    nvt = torch.tensor(nv, dtype=torch.int64, device=DEV)
    idx, _ = C.csa2_topk(s, nvt, 512, pool=pool)
    idx, sn, pl = to_np(idx), s.double().cpu().numpy(), to_np(pool)
    for r in range(rows):
        full = np.full(max(nv[r], 1), -np.inf)
        for c_ in range(n_pool * 8):
            b = pl[r, c_ // 8]
            e = int(b) * 8 + c_ % 8
            if b >= 0 and e < nv[r]:
                full[e] = sn[r, c_]
        ref = O.reindex_topk(full, pl[r], nv[r], 512)
        np.testing.assert_array_equal(idx[r], ref, err_msg=f"row {r}")


@pytest.mark.parametrize("pos", [0, 1, 4095, 131072, (1 << 20) - 1, (1 << 31) - 7])
def test_rope_angles_at_large_positions(pos):
    """The write epilogue's RoPE (m = 1: the entry is its token, rotated at its
    position) against the oracle's f64 angles, to 2e-6 of the row scale."""
    B = 4
    C_ = W.normal_tensor((B, 1, 512), 181, 1, torch.float32, DEV)
    Z_ = W.normal_tensor((B, 1, 512), 181, 2, torch.float32, DEV)
    pos0 = torch.tensor([pos, pos + 1, pos // 3, 7], dtype=torch.int64, device=DEV)
    out = C.csa2_compress(C_, Z_, 1, pos0=pos0, flags=C.W_ROPE, out_fmt="f32")
    for b in range(B):
        ref = O.rope(C_[b, 0].double().cpu().numpy(), int(pos0[b]))
        np.testing.assert_allclose(to_np(out)[b, 0], ref, rtol=0, atol=2e-6 * np.abs(ref).max())


@pytest.mark.parametrize("V", [1, 9, 4000, 4097, 8 * 2048, 8 * 2048 + 1, 262143])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("k", [100, 512, 1024])
def test_pool_topk_bit_exact(V, ties, k):
    """csa2_pool_topk: the pool and the top-k entries from block maxima, their
    histogram and the full scores -- both bit-exact with the oracle's block_pool and
    topk over the same scores, ties and crowded threshold bins included."""
    N = 262144
    s = _score_rows(3, N, 81 + V, ties)
    nv = torch.tensor([V, max(V - 7, 0), min(V + 3, N)], dtype=torch.int64, device=DEV)
    sn = s.double().cpu().numpy()
    # the block maxima are the oracle's own; the library summarises them
    bm = torch.tensor(np.stack([O.block_max(np.where(np.arange(N) < int(nv[r]), sn[r], -np.inf), N, 8)
                                for r in range(3)]), dtype=torch.float32, device=DEV)
    hist = C.csa2_block_hist(bm, nv, 8)
    pool, idx, val = C.csa2_pool_topk(bm, hist, s, nv, k, want_scores=True)
    C.csa2_ctx_check()
    for r in range(3):
        Vr = int(nv[r])
        np.testing.assert_array_equal(to_np(pool)[r], O.block_pool(O.block_max(sn[r], Vr, 8), Vr, 8, 2048))
        ref = O.topk(sn[r], Vr, k)
        np.testing.assert_array_equal(to_np(idx)[r], ref, err_msg=f"row {r} V {Vr}")
        np.testing.assert_array_equal(to_np(val)[r], np.where(ref >= 0, sn[r][np.maximum(ref, 0)], -np.inf))



@pytest.mark.parametrize("order", ["rising", "falling", "random"])
def test_pool_topk_blocks_of_one_many_winners(order):
    """Blocks of one entry and k = 3,000: with rising scores every winner lies in the
    last CTA's chunk (more winners than one CTA lists, so they are emitted from its
    bitmap), with falling scores in the first, at random everywhere; pool and top-k
    bit-exact with the oracle, equal scores included."""
    N, k, n_keep = 131072, 3000, 4096
    g = torch.Generator().manual_seed(7)
    base = torch.arange(N, dtype=torch.float64)
    if order == "falling":
        base = -base
    elif order == "random":
        base = torch.randn(N, generator=g, dtype=torch.float64)
    sc = torch.floor(base * 4) / 4                       # many equal scores
    s = sc.to(torch.float32).view(1, N).to(DEV)
    nv = torch.tensor([N - 5], dtype=torch.int64, device=DEV)
    sn = s.double().cpu().numpy()[0]
    V = int(nv[0])
    bm = torch.tensor(O.block_max(np.where(np.arange(N) < V, sn, -np.inf), N, 1), dtype=torch.float32,
                      device=DEV).view(1, N)
    hist = C.csa2_block_hist(bm, nv, 1)
    pool, idx, val = C.csa2_pool_topk(bm, hist, s, nv, k, block=1, n_keep=n_keep, want_scores=True)
    C.csa2_ctx_check()
    np.testing.assert_array_equal(to_np(pool)[0], O.block_pool(O.block_max(sn, V, 1), V, 1, n_keep))
    ref = O.topk(sn, V, k)
    np.testing.assert_array_equal(to_np(idx)[0], ref)
    np.testing.assert_array_equal(to_np(val)[0], sn[ref])


def test_pool_topk_rejects_too_many_candidates():
    """k * block above the receive capacity (8,192 entries) is refused on the host (the
    decode step then takes the pool, the best blocks' rescoring and csa2_topk one by
    one)."""
    N = 16384
    s = _score_rows(1, N, 91, False)
    nv = torch.tensor([N], dtype=torch.int64, device=DEV)
    bm = torch.zeros((1, N // 8), dtype=torch.float32, device=DEV)
    hist = C.csa2_block_hist(bm, nv, 8)
    with pytest.raises(C.Csa2Error):
        C.csa2_pool_topk(bm, hist, s, nv, 1100)


def test_visible_entries_causal_rule():
    """floor(t / m) per query position, the oracle's visibility rule, over positions
    around every block edge, far positions and negative ones (which see nothing)."""
    pos = [-5, -1, 0, 1, 3, 4, 5, 127, 128, 129, 4095, 4096, 1 << 20, (1 << 20) - 1, (1 << 40) + 3]
    for m in (1, 2, 4, 128):
        t = torch.tensor(pos, dtype=torch.int64, device="cuda")
        nv = C.csa2_visible_entries(t.view(3, 5), m)
        C.csa2_ctx_check()
        ref = [O.visible_entries(p, m) if p >= 0 else 0 for p in pos]
        assert nv.view(-1).cpu().tolist() == ref, m
        # in place
        C.csa2_visible_entries(t, m, out=t)
        assert t.cpu().tolist() == ref
    with pytest.raises(ValueError):
        C.csa2_visible_entries(torch.zeros(3, dtype=torch.int32, device="cuda"), 2)
