"""Pins for the oracle's indexer score, visibility, top-k and block pool."""
import itertools

import numpy as np
import pytest

from oracle import csa2_oracle as O


def test_worked_example_scores_and_ids(golden):
    g = golden("sparse_shared_kv_example.json")
    sc = O.index_score(np.array(g["iq"]), np.array(g["head_weight"]), np.array(g["ik"]), 3)
    np.testing.assert_array_equal(sc, np.array(g["hand_derived"]["scores"]))
    ids = O.topk(sc, 3, g["k"])
    assert 2 in ids.tolist()                               # what the page asserts
    np.testing.assert_array_equal(ids, g["hand_derived"]["ids_ascending"])


def test_index_score_brute_force_loops():
    r = np.random.default_rng(1)
    H, d, N, V = 5, 7, 23, 19
    qI, KI, w = r.normal(size=(H, d)), r.normal(size=(N, d)), r.normal(size=H)
    sc = O.index_score(qI, w, KI, V)
    for s in range(N):
        if s >= V:
            assert sc[s] == -np.inf
            continue
        tot = 0.0
        for h in range(H):
            dot = 0.0
            for j in range(d):
                dot += qI[h, j] * KI[s, j]
            tot += w[h] * (dot if dot > 0 else 0.0)
        assert sc[s] == pytest.approx(tot, rel=1e-12, abs=1e-12)


def test_index_score_sign_properties():
    r = np.random.default_rng(2)
    qI, KI = r.normal(size=(4, 8)), r.normal(size=(50, 8))
    assert np.all(O.index_score(qI, -np.abs(r.normal(size=4)), KI, 50) <= 0)
    assert np.all(O.index_score(qI, np.abs(r.normal(size=4)), KI, 50) >= 0)
    # keys opposite to every query head: all ReLUs are 0, so all scores are 0 and
    # the lowest indices win
    qI = np.abs(r.normal(size=(4, 8)))
    KI = -np.abs(r.normal(size=(50, 8)))
    sc = O.index_score(qI, r.normal(size=4), KI, 50)
    assert np.all(sc == 0)
    np.testing.assert_array_equal(O.topk(sc, 50, 10), np.arange(10))


def test_visibility_rule():
    # DSA-to-CSA/HCA page: with m' = 128, position 127 cannot read entry 0,
    # position 128 can.
    assert O.visible_entries(100, 128) == 0
    assert O.visible_entries(127, 128) == 0
    assert O.visible_entries(128, 128) == 1
    assert O.visible_entries(4095, 2) == 2047 and O.visible_entries(4092, 2) == 2046
    assert O.visible_entries(65535, 1) == 65535


def _brute_topk(s, V, k):
    order = sorted(range(V), key=lambda i: (-s[i], i))
    sel = sorted(order[:k])
    return sel + [-1] * (k - len(sel))


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    r = np.random.default_rng(seed)
    N = 200
    s = r.integers(-5, 6, size=N).astype(float)           # heavy ties
    for V in (0, 1, 7, 31, 32, 33, 150, 200):
        for k in (1, 16, 32, 64):
            assert O.topk(s, V, k).tolist() == _brute_topk(s, V, k)


def test_topk_edge_cases():
    s = np.full(1000, 3.5)
    np.testing.assert_array_equal(O.topk(s, 1000, 512), np.arange(512))   # all equal
    out = O.topk(np.arange(10.0), 10, 512)                                 # fewer than k
    assert out[:10].tolist() == list(range(10)) and np.all(out[10:] == -1)
    assert np.all(O.topk(np.arange(10.0), 0, 8) == -1)                     # none visible
    # -0.0 and +0.0 are equal scores: the lower index wins
    s = np.array([0.0, -0.0, -0.0, 0.0, -1.0])
    assert O.topk(s, 5, 2).tolist() == [0, 1]


def _brute_pool(bm, V, block, n_keep):
    if V == 0:
        return [-1] * n_keep
    nb = (V + block - 1) // block
    b_new = (V - 1) // block
    if nb <= n_keep:
        return list(range(nb)) + [-1] * (n_keep - nb)
    others = sorted((b for b in range(nb) if b != b_new), key=lambda b: (-bm[b], b))
    return sorted(others[: n_keep - 1] + [b_new])


@pytest.mark.parametrize("seed", range(5))
def test_block_max_and_pool_brute_force(seed):
    r = np.random.default_rng(seed)
    N = 300
    s = r.integers(-3, 4, size=N).astype(float)
    for V in (0, 1, 8, 9, 63, 64, 65, 299):
        bm = O.block_max(s, V, 8)
        nb = (V + 7) // 8
        assert len(bm) == nb
        for b in range(nb):
            assert bm[b] == max(s[8 * b: min(8 * b + 8, V)])
        for n_keep in (1, 2, 4, 8, 40):
            assert O.block_pool(bm, V, 8, n_keep).tolist() == _brute_pool(bm, V, 8, n_keep)


def test_newest_block_always_kept():
    s = np.concatenate([np.full(64, 100.0), np.full(17, -100.0)])
    V = 81
    pool = O.block_pool(O.block_max(s, V, 8), V, 8, 4)
    assert (V - 1) // 8 in pool.tolist()                  # partial block 10 kept
    assert pool.tolist() == [0, 1, 2, 10]


@pytest.mark.parametrize("seed", range(8))
def test_lemma_topk_inside_pool(seed):
    # With one (score desc, index asc) order, the top-k entries lie inside the
    # pool of the best n_keep blocks when n_keep - 1 >= k.
    r = np.random.default_rng(seed)
    N = 4000
    s = np.round(r.normal(size=N) * 2) / 2                 # many ties
    for V, k, n_keep in ((3999, 40, 41), (3999, 64, 100), (2000, 16, 17), (500, 100, 101)):
        ids = O.topk(s, V, k)
        pool = O.block_pool(O.block_max(s, V, 8), V, 8, n_keep)
        cand = set(O.pool_candidates(pool, V, 8).tolist())
        assert set(i for i in ids.tolist() if i >= 0) <= cand
        # and re-selecting inside the pool gives the same top-k
        np.testing.assert_array_equal(O.reindex_topk(s, pool, V, k), ids)


def test_reindex_with_all_blocks_is_full_topk():
    r = np.random.default_rng(11)
    s = r.normal(size=1000)
    V = 997
    pool = np.arange((V + 7) // 8)
    np.testing.assert_array_equal(O.reindex_topk(s, pool, V, 64), O.topk(s, V, 64))


def test_reindex_candidates_only():
    s = np.arange(100, dtype=float)                        # later entries score higher
    pool = np.array([1, 3, -1, -1])
    V = 30                                                 # block 3 is partial: 24..29
    ids = O.reindex_topk(s, pool, V, 5)
    assert ids.tolist() == [25, 26, 27, 28, 29]
    ids = O.reindex_topk(s, pool, V, 20)
    assert ids.tolist() == list(range(8, 16)) + list(range(24, 30)) + [-1] * 6


def test_merge_topk_over_entry_shards():
    r = np.random.default_rng(12)
    s = np.round(r.normal(size=3000) * 3) / 3
    V, k = 2990, 100
    full = O.topk(s, V, k)
    edges = [0, 700, 1500, 2990]
    ids, scs = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        loc = O.topk(s[a:b], b - a, k)
        g = np.where(loc >= 0, loc + a, -1)
        ids.append(g)
        scs.append(np.where(g >= 0, s[np.maximum(g, 0)], -np.inf))
    np.testing.assert_array_equal(O.merge_topk(ids, scs, k), full)


def test_planted_keys_of_the_bf16_decode_workload_are_selected():
    """The bf16 decode workload plants 16 keys per sequence along the direction of the
    positively weighted indexer heads (about twelve times a random key's length): on
    the oracle they score at least 8 standard deviations above the mean, sit in the
    top-512 and their blocks in the 2,048-block pool (DSA-to-CSA/HCA eqs. (16)-(17);
    CSA2 page «解码器里的分层索引»).  Two sequences at the workload's 64K entries."""
    from compressed_sparse_attention_06_gb300 import workloads as W
    wl = W.decode_full_bf16("cpu", B=2, N=65536, with_main_kv=False)
    t = wl.tensors
    V = wl.N - 1
    for b in range(2):
        sc = O.index_score(t["qI"][b, 0].double().numpy(), t["w"][b, 0].double().numpy(),
                           t["KI"][b].double().numpy(), V)
        planted = t["planted"][b].numpy()
        vis = sc[:V]
        assert np.all(sc[planted] >= vis.mean() + 8 * vis.std())
        assert set(planted.tolist()) <= set(O.topk(sc, V, 512).tolist())
        assert set((planted // 8).tolist()) <= set(O.block_pool(O.block_max(sc, V, 8), V, 8, 2048).tolist())
