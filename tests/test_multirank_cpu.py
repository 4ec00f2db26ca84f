"""World-size-2 gloo ranks on CPU: the multi-GPU host logic.  Each rank scores its
entry range and attends over its share of the keys with the oracle; the merged
result must equal the unsharded oracle result.  Also the per-rank sequence split
and the max-over-ranks timing reduction."""
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
