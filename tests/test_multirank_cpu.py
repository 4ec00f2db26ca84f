"""gloo ranks on CPU: the multi-GPU host logic.  Each rank scores its entry range
and attends over its share of the keys with the oracle; the merged result must
equal the unsharded oracle result.  The pooled decode step is sharded the same
way: each rank keeps its own block pool (block ids + block maxima) and its own
top-k inside that pool, one all-gather of those keys, and the merged pool and
top-k must equal the unsharded ones (CSA2 page, «解码器里的分层索引»).  Also the
per-rank sequence split and the max-over-ranks timing reduction."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from compressed_sparse_attention_06_gb300 import sharding as S
from oracle import csa2_oracle as O


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    r = np.random.default_rng(5)
    N, H_I, H, c, k = 3000, 8, 4, 64, 100
    return dict(qI=r.normal(size=(H_I, 128)), w=r.normal(size=H_I), KI=np.round(r.normal(size=(N, 128)) * 2) / 2,
                q=r.normal(size=(H, c)), kv=r.normal(size=(N, c)), swa=r.normal(size=(16, c)),
                sink=r.normal(size=H), V=2990, t=2990, k=k)


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = _problem()
        lo, hi = S.entry_range(rank, world, p["V"])
        sc = O.index_score(p["qI"], p["w"], p["KI"][lo:hi], hi - lo)
        loc = O.topk(sc, hi - lo, p["k"])
        ids = torch.from_numpy(np.where(loc >= 0, loc + lo, -1))
        scs = torch.from_numpy(np.where(loc >= 0, sc[np.maximum(loc, 0)], -np.inf))
        g_ids = [torch.zeros_like(ids) for _ in range(world)]
        g_scs = [torch.zeros_like(scs) for _ in range(world)]
        dist.all_gather(g_ids, ids)
        dist.all_gather(g_scs, scs)
        merged = S.merge_topk(g_ids, g_scs, p["k"]).numpy()
        # attention: this rank's share of the selected rows; the window goes to rank 0
        mine = [i for i in merged if i >= 0 and lo <= i < hi]
        keys = [p["kv"][i] for i in mine]
        if rank == 0:
            keys += [p["swa"][pp % 16] for pp in range(p["t"] - 15, p["t"] + 1)]
        o, lse, _ = O.attend(p["q"], np.array(keys).reshape(len(keys), -1), p["t"], None)
        g_o = [torch.zeros((4, 64), dtype=torch.float64) for _ in range(world)]
        g_l = [torch.zeros(4, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(g_o, torch.from_numpy(o))
        dist.all_gather(g_l, torch.from_numpy(lse))
        om, lm = S.merge_attention(g_o, g_l, torch.from_numpy(p["sink"]))
        slowest = S.max_over_ranks(1.0 + rank)
        seq0, nseq = S.sequences_for_rank(rank, world, 8)
        q.put((rank, merged, om.numpy(), lm.numpy(), slowest, seq0, nseq))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_merge_exactly():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    res.sort(key=lambda x: x[0])
    p = _problem()
    full_sc = O.index_score(p["qI"], p["w"], p["KI"], p["V"])
    ref_ids = O.topk(full_sc, p["V"], p["k"])
    keys = np.concatenate([p["kv"][[i for i in ref_ids if i >= 0]],
                           p["swa"][[pp % 16 for pp in range(p["t"] - 15, p["t"] + 1)]]])
    o_ref, l_ref, _ = O.attend(p["q"], keys, p["t"], p["sink"])
    for rank, merged, om, lm, slowest, seq0, nseq in res:
        np.testing.assert_array_equal(merged, ref_ids)
        np.testing.assert_allclose(om, o_ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lm, l_ref, rtol=1e-13)
        assert slowest == 2.0
        assert (seq0, nseq) == (8 * rank, 8)


def test_entry_ranges_cover_exactly():
    for n in (0, 1, 7, 1000, 1 << 20):
        for world in (1, 2, 3, 8):
            rs = [S.entry_range(r, world, n) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(rs[:-1], rs[1:]))
            assert max(h - l for l, h in rs) - min(h - l for l, h in rs) <= 1


def _pool_problem(ties):
    """One long sequence for the pooled step.  ties=True puts the indexer inputs on a
    coarse grid (many equal scores and equal block maxima across ranks)."""
    r = np.random.default_rng(11 if ties else 12)
    N, H_I, H, c = 20000, 8, 4, 64
    qI, KI, w = r.normal(size=(H_I, 128)), r.normal(size=(N, 128)), r.normal(size=H_I)
    if ties:
        qI, KI, w = np.round(qI), np.round(KI * 0.5), np.sign(w)
    return dict(qI=qI, w=w, KI=KI, q=r.normal(size=(H, c)), kv=r.normal(size=(N, c)), swa=r.normal(size=(16, c)),
                sink=r.normal(size=H), N=N, V=19995, t=19995, k=60, n_keep=96)


def _rank_pool_main(rank, world, port, ties, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = _pool_problem(ties)
        k, n_keep, V = p["k"], p["n_keep"], p["V"]
        lo, hi = S.entry_range(rank, world, p["N"], align=8)
        V_r = max(0, min(V - lo, hi - lo))
        # this rank's share of the step (the oracle stands in for the library on CPU)
        sc = O.index_score(p["qI"], p["w"], p["KI"][lo:hi], V_r)
        bm = O.block_max(sc, V_r, 8)
        pool = O.block_pool(bm, V_r, 8, n_keep)
        top = O.reindex_topk(sc, pool, V_r, k) if V_r else np.full(k, -1)
        pool_ids = torch.from_numpy(np.where(pool >= 0, pool + lo // 8, -1))
        pool_max = torch.from_numpy(np.where(pool >= 0, bm[np.maximum(pool, 0)] if len(bm) else 0.0, -np.inf))
        top_ids = torch.from_numpy(np.where(top >= 0, top + lo, -1))
        top_sc = torch.from_numpy(np.where(top >= 0, sc[np.maximum(top, 0)], -np.inf))
        gathered = []
        for t in (pool_ids, pool_max, top_ids, top_sc):          # one all-gather of n_keep + k keys
            g = [torch.zeros_like(t) for _ in range(world)]
            dist.all_gather(g, t)
            gathered.append(g)
        pool_m = S.merge_pool(gathered[0], gathered[1], V, 8, n_keep).numpy()
        top_m = S.merge_topk(gathered[2], gathered[3], k).numpy()
        # attention over this rank's share of the merged selection; the window on the last rank
        keys = [p["kv"][i] for i in top_m if i >= 0 and lo <= i < hi]
        if rank == world - 1:
            keys += [p["swa"][pp % 16] for pp in range(p["t"] - 15, p["t"] + 1)]
        o, lse, _ = O.attend(p["q"], np.array(keys).reshape(len(keys), -1), p["t"], None)
        g_o = [torch.zeros((4, 64), dtype=torch.float64) for _ in range(world)]
        g_l = [torch.zeros(4, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(g_o, torch.from_numpy(o))
        dist.all_gather(g_l, torch.from_numpy(lse))
        om, lm = S.merge_attention(g_o, g_l, torch.from_numpy(p["sink"]))
        q.put((rank, pool_m, top_m, om.numpy(), lm.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("ties", [False, True], ids=["gaussian", "ties"])
def test_gloo_ranks_pooled_decode_merges_exactly(world, ties):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_pool_main, args=(r, world, port, ties, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=180) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    p = _pool_problem(ties)
    V, k, n_keep = p["V"], p["k"], p["n_keep"]
    full = O.index_score(p["qI"], p["w"], p["KI"], V)
    pool_ref = O.block_pool(O.block_max(full, V, 8), V, 8, n_keep)
    top_ref = O.topk(full, V, k)
    if ties:   # the tie-heavy problem really has tied block maxima at the pool's cut
        bm = O.block_max(full, V, 8)
        assert len(set(bm[pool_ref[pool_ref >= 0]].tolist()) & set(np.delete(bm, pool_ref).tolist())) > 0
    keys = np.concatenate([p["kv"][[i for i in top_ref if i >= 0]],
                           p["swa"][[pp % 16 for pp in range(p["t"] - 15, p["t"] + 1)]]])
    o_ref, l_ref, _ = O.attend(p["q"], keys, p["t"], p["sink"])
    for rank, pool_m, top_m, om, lm in res:
        np.testing.assert_array_equal(pool_m, pool_ref)
        np.testing.assert_array_equal(top_m, top_ref)
        np.testing.assert_allclose(om, o_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lm, l_ref, rtol=1e-13)


def test_merge_pool_edge_cases():
    """Few visible blocks keep them all; V = 0 keeps none; the newest block is kept
    even when it scores lowest; ties go to the lower block id."""
    assert S.merge_pool([torch.tensor([0, 1, -1])], [torch.tensor([1.0, 2.0, -np.inf])], 12, 8, 4).tolist() == \
        [0, 1, -1, -1]
    assert S.merge_pool([torch.tensor([-1])], [torch.tensor([-np.inf])], 0, 8, 4).tolist() == [-1] * 4
    ids = [torch.tensor([0, 1, 2]), torch.tensor([3, 4, 5])]
    mx = [torch.tensor([5.0, 7.0, 7.0]), torch.tensor([7.0, 1.0, -3.0])]
    # 6 blocks, V = 48 -> newest block 5; keep 3: block 5 plus the best two others (7.0 ties: 1, 2 before 3)
    assert S.merge_pool(ids, mx, 48, 8, 3).tolist() == [1, 2, 5]


def test_aligned_entry_ranges():
    for n in (0, 5, 8, 1000, 20000, (1 << 20) - 1):
        for world in (1, 2, 3, 8):
            rs = [S.entry_range(r, world, n, align=8) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(rs[:-1], rs[1:]))
            assert all(lo % 8 == 0 for lo, hi in rs if hi > lo)      # empty ranges sit at n
