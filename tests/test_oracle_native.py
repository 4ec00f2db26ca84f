"""The C++ restatement of the oracle (oracle/csa2_oracle.cpp) against the pages'
worked examples and against the numpy oracle, on pinned examples and small random
inputs.  No GPU: the library is built with the host compiler."""
import math
import shutil

import numpy as np
import pytest

from oracle import csa2_oracle as O

if shutil.which("g++") is None:
    pytest.skip("no host C++ compiler", allow_module_level=True)

from oracle import native as NO  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    NO.build()
    assert NO.lib().csa2o_version() == 1


def _dyadic(r, shape, lo=-8, hi=8, den=8):
    """Values on a grid of 1/den: every product and short sum below is exact in f64,
    so both oracles reach the same bits whatever their summation order."""
    return r.integers(lo * den, hi * den + 1, size=shape) / den


# ---------------------------------------------------------------- the pages' examples
def test_worked_example_indexer_and_attention(golden):
    g = golden("sparse_shared_kv_example.json")
    hd = g["hand_derived"]
    sc = NO.index_score(np.array(g["iq"]), np.array(g["head_weight"]), np.array(g["ik"]), 3)
    np.testing.assert_array_equal(sc, hd["scores"])
    ids = NO.topk(sc, 3, g["k"])
    np.testing.assert_array_equal(ids, hd["ids_ascending"])
    o, lse = NO.sparse_attn(np.array([g["q"]]), np.array(g["kv"]), ids, np.zeros((1, 2)), 0, 0,
                            sink=np.array([g["sink_logit"]]), window=0, flags=0)
    np.testing.assert_allclose(o[0], hd["out"], rtol=1e-9)
    a, b = math.exp(math.sqrt(2)), math.exp(1 / math.sqrt(2))
    np.testing.assert_allclose(lse[0], math.log(a + b + 1), rtol=1e-14)


def test_worked_example_compressor(golden):
    g = golden("compressor_worked_example.json")
    m, c = g["m"], g["c"]
    Ca = np.array(g["Ca_rows"], dtype=float)
    Cb = np.array(g["Cb_rows"], dtype=float)
    Z = np.zeros_like(Ca)
    y = NO.compress(Ca, Z, m, np.zeros((m, c)), Cb, Z, np.zeros((m, c)))
    np.testing.assert_allclose(y, np.array(g["expected"]), rtol=0, atol=1e-15)


def test_code_tables(golden):
    g = golden("fp4_code_tables.json")
    vals = np.array([NO.e2m1_value(i) for i in range(16)])
    exp = np.array(g["e2m1_values_by_code"])
    np.testing.assert_array_equal(vals, exp)
    np.testing.assert_array_equal(np.signbit(vals), np.signbit(exp))
    for k, v in g["e4m3_selected"].items():
        assert NO.e4m3_value(int(k, 16)) == v, k
    for k, v in g["e8m0_selected"].items():
        assert NO.e8m0_value(int(k)) == v, k
    e4 = np.array([NO.e4m3_value(i) for i in range(256)])
    np.testing.assert_array_equal(e4, O.e4m3_decode(np.arange(256)))
    e8 = np.array([NO.e8m0_value(i) for i in range(256)])
    np.testing.assert_array_equal(e8, O.e8m0_decode(np.arange(256)))


def test_encoders_agree_on_ties_and_saturation(golden):
    g = golden("fp4_code_tables.json")
    r = np.random.default_rng(3)
    grid = O.e2m1_decode(np.arange(8))
    mids = (grid[1:] + grid[:-1]) / 2
    xs = np.concatenate([grid, -grid, mids, -mids, [0.0, -0.0, 7.0, -1e9, 1e9, 5.999, 6.001],
                         r.normal(size=300) * 4])
    for x in xs:
        assert NO.e2m1_encode(x) == int(O.e2m1_encode(x)), x
    e4 = O.e4m3_decode(np.arange(0x7F))
    xs = np.concatenate([e4, (e4[1:] + e4[:-1]) / 2, [500.0, 1e6, -0.0], r.lognormal(size=300) * 0.01])
    for x in xs:
        assert NO.e4m3_encode(x) == int(O.e4m3_encode(x)), x
        assert NO.e4m3_encode(-x) == int(O.e4m3_encode(-x)), x


# ---------------------------------------------------------------- formats
def _fp4_rows(r, rows, c):
    x = (r.normal(size=(rows, c)) * r.lognormal(sigma=2.0, size=(rows, 1))).astype(np.float32)
    x[0, :32] = 0.0                                     # an all-zero scale group
    x[1, 16:48] = 1e30                                  # saturating groups
    x[2, 3] = -0.0
    return x


def test_nvfp4_pack_bytes_and_unpack():
    r = np.random.default_rng(4)
    x = _fp4_rows(r, 64, 512)
    b = NO.nvfp4_pack(x)
    np.testing.assert_array_equal(b, O.nvfp4_pack(x))
    np.testing.assert_array_equal(NO.nvfp4_unpack(b), O.nvfp4_unpack(b))


def test_mxfp4_pack_bytes_and_unpack():
    r = np.random.default_rng(5)
    x = _fp4_rows(r, 64, 128)
    x[3, :32] = 2.0 ** -140                             # scale exponent clamped at 0
    b = NO.mxfp4_pack(x)
    np.testing.assert_array_equal(b, O.mxfp4_pack(x))
    np.testing.assert_array_equal(NO.mxfp4_unpack(b), O.mxfp4_unpack(b))


# ---------------------------------------------------------------- compressor, norm, RoPE
@pytest.mark.parametrize("overlap", [False, True])
def test_compress_random(overlap):
    r = np.random.default_rng(6)
    m, c, n = 4, 24, 20
    Ca, Za, Cb, Zb = (r.normal(size=(n, c)) for _ in range(4))
    Ba, Bb, pC, pZ = (r.normal(size=(m, c)) for _ in range(4))
    if overlap:
        got = NO.compress(Ca, Za, m, Ba, Cb, Zb, Bb, pC, pZ)
        ref = O.compress(Ca, Za, m, Ba, Cb, Zb, Bb, pC, pZ)
        np.testing.assert_allclose(NO.compress(Ca, Za, m, Ba, Cb, Zb, Bb), O.compress(Ca, Za, m, Ba, Cb, Zb, Bb),
                                   rtol=1e-13, atol=1e-14)
    else:
        got, ref = NO.compress(Ca, Za, m, Ba), O.compress(Ca, Za, m, Ba)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_norm_rope_and_write_epilogue():
    r = np.random.default_rng(7)
    x = r.normal(size=(5, 512)) * 3
    np.testing.assert_allclose(NO.rms_norm(x), O.rms_norm(x), rtol=1e-14)
    # the angle pos * theta carries about pos * ulp(theta) of rounding on either side
    # (the two libraries' pow may differ in the last bit; theta <= 1), so the rotated
    # values agree to |x| * 4 * pos * 2^-52
    for pos, inv in [(0, False), (7, False), (1_048_575, True), (4_194_303, False), (123_456_789, False)]:
        tol = 1e-13 + np.abs(x).max() * 4 * pos * 2.0 ** -52
        np.testing.assert_allclose(NO.rope(x, pos, inv), O.rope(x, pos, inv), rtol=0, atol=tol)
    for flags in (1, 2, 3):
        np.testing.assert_allclose(NO.compress_write(x, flags, 4, pos0=3), O.compress_write(x, flags, 4, pos0=3),
                                   rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- indexer and selection
def test_index_score_exact_on_a_dyadic_grid():
    r = np.random.default_rng(8)
    qI, w, K = _dyadic(r, (6, 32)), _dyadic(r, 6), _dyadic(r, (50, 32))
    for V in (0, 1, 37, 50):
        np.testing.assert_array_equal(NO.index_score(qI, w, K, V), O.index_score(qI, w, K, V))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topk_block_pool_reindex_with_ties(seed):
    r = np.random.default_rng(seed)
    N = 300
    sc = r.integers(0, 12, size=N).astype(float)        # many ties
    for V in (0, 1, 5, 64, 299, 300):
        for k in (1, 16, 64):
            np.testing.assert_array_equal(NO.topk(sc, V, k), O.topk(sc, V, k))
        for block in (1, 8, 16):
            bm = NO.block_max(sc, V, block)
            np.testing.assert_array_equal(bm, O.block_max(sc, V, block))
            for n_keep in (2, 5, 40):
                pool = NO.block_pool(bm, V, block, n_keep)
                np.testing.assert_array_equal(pool, O.block_pool(bm, V, block, n_keep))
                np.testing.assert_array_equal(NO.reindex_topk(sc, pool, V, 16, block),
                                              O.reindex_topk(sc, pool, V, 16, block))


# ---------------------------------------------------------------- attention
@pytest.mark.parametrize("flags", [0, O.QNORM | O.KVNORM | O.ROPE, O.KVNORM])
def test_sparse_attn_random(flags):
    r = np.random.default_rng(9)
    H, c, N, cap = 4, 128, 40, 16
    q, kv, swa = r.normal(size=(H, c)), r.normal(size=(N, c)), r.normal(size=(cap, c))
    idx = np.array([3, 7, -1, 20, 39, -1])
    sink = r.normal(size=H)
    for t, window, s in [(500, 8, sink), (3, 16, None), (40, 0, sink), (100, 16, None)]:
        o, lse = NO.sparse_attn(q, kv, idx, swa, 5, t, s, window, flags)
        o_ref, lse_ref, _ = O.sparse_attn(q, kv, idx, swa, 5, t, s, window, flags)
        np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


def test_decode_query_fp4_matches_the_numpy_pipeline():
    """The threaded decode baseline against the numpy oracle's steps: MXFP4 dequant,
    scores, block max, pool, top-k inside the pool, FP4 rows, attention."""
    r = np.random.default_rng(10)
    N, H_I, H, k, block, n_keep, window = 3000, 8, 4, 32, 8, 24, 16
    ki = NO.mxfp4_pack(r.normal(size=(N, 128)).astype(np.float32))
    qI_mx = NO.mxfp4_pack(r.normal(size=(H_I, 128)).astype(np.float32))
    w = _dyadic(r, H_I, 0, 2)
    kv_f = r.normal(size=(N, 512)).astype(np.float32)
    kv = NO.nvfp4_pack(kv_f)
    q, swa, sink = r.normal(size=(H, 512)), r.normal(size=(window, 512)), r.normal(size=H)
    for V, t in [(N, N + 5), (2999, 2999), (100, 100), (5, 5)]:
        o, lse, idx = NO.decode_query_fp4(ki, V, qI_mx, w, np.arange(N), kv, q, swa, 0, t, sink, block=block,
                                          n_keep=n_keep, k=k, window=window, threads=3)
        sc = O.index_score(O.mxfp4_unpack(qI_mx), w, O.mxfp4_unpack(ki), V)
        pool = O.block_pool(O.block_max(sc, V, block), V, block, n_keep)
        idx_ref = O.reindex_topk(sc, pool, V, k, block)
        np.testing.assert_array_equal(idx, idx_ref)
        o_ref, lse_ref, _ = O.sparse_attn(q, O.nvfp4_unpack(kv), idx_ref, swa, 0, t, sink, window)
        np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)
    # only the selected rows need to be handed over
    sel = idx[idx >= 0]
    o2, _, idx2 = NO.decode_query_fp4(ki, 5, qI_mx, w, sel, kv[sel], q, swa, 0, 5, sink, block=block, n_keep=n_keep,
                                      k=k, window=window, threads=2)
    np.testing.assert_array_equal(idx2, idx)
    np.testing.assert_array_equal(o2, o)
    with pytest.raises(ValueError):
        NO.decode_query_fp4(ki, 5, qI_mx, w, sel[1:], kv[sel[1:]], q, swa, 0, 5, sink, block=block,
                            n_keep=n_keep, k=k, window=window, threads=2)
