"""The pooled decode step sharded by entry range, through the library: each rank's
share (sharding.rank_select / rank_attention on the rows it holds) runs as its own
library calls, one rank after another on this GPU (the calls never wait on each
other), the per-rank results are stacked as an all-gather would deliver them, and
the host merges must give exactly the unsharded step's pool and top-k, and its
attention up to rounding (CSA2 page, «解码器里的分层索引»)."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import pipeline as P
from compressed_sparse_attention_06_gb300 import sharding as S
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _caches(B, N):
    kv = torch.empty((B, N, 288), dtype=torch.uint8, device=DEV)
    ki = torch.empty((B, N, 68), dtype=torch.uint8, device=DEV)
    for b in range(B):
        C.csa2_fp4_pack(W.fp4_rows("kv", b, 0, N, N, DEV), C.FP4_E4M3x16, out=kv[b])
        C.csa2_fp4_pack(W.fp4_rows("KI", b, 0, N, N, DEV), C.MXFP4_E8M0x32, out=ki[b])
    return kv, ki


@pytest.mark.parametrize("world", [2, 3, 5])
def test_sharded_pooled_decode_equals_unsharded(world):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    B, N, H = 2, 1 << 18, 64
    wl = W.fp4_decode(DEV, B=B, N=N, H=H)
    kv, ki = _caches(B, N)
    q_pos = torch.tensor([[N - 1], [N - 5000]], dtype=torch.int64, device=DEV)
    nv = P.visible_entries(q_pos, 1)
    buf = P.alloc_decode(B, 1, N, H, 512, DEV, out_dtype=torch.float32)
    P.full_decode_step(wl["qI"], wl["w"], ki, wl["q"], kv, wl["swa"], q_pos, nv, wl["sink"], buf)
    parts, atts = [], []
    ranges = [S.entry_range(r, world, N, align=8) for r in range(world)]
    for lo, hi in ranges:                          # each rank holds only its own rows
        parts.append(S.rank_select(wl["qI"], wl["w"], ki[:, lo:hi].contiguous(), lo, nv))
    pool_m, top_m = S.merge_selections(parts, nv.cpu())
    for r, (lo, hi) in enumerate(ranges):
        atts.append(S.rank_attention(wl["q"], kv[:, lo:hi].contiguous(), lo, top_m, wl["swa"], q_pos,
                                     with_window=(r == world - 1)))
    C.csa2_ctx_check()
    np.testing.assert_array_equal(pool_m.numpy(), to_np(buf.pool).astype(np.int64))
    np.testing.assert_array_equal(top_m.numpy(), to_np(buf.idx).astype(np.int64))
    for b in range(B):
        o, lse = S.merge_attention([a[0][b, 0].cpu() for a in atts], [a[1][b, 0].cpu() for a in atts],
                                   wl["sink"].cpu())
        assert_close(o.numpy(), to_np(buf.out[b, 0]), 5e-3, f"b{b}: merged vs unsharded attention")
        # and against the oracle's attention over the same selection
        t = int(q_pos[b, 0])
        sel = top_m[b, 0].numpy()
        rows = {int(s): O.nvfp4_unpack(O.nvfp4_pack(W.fp4_rows("kv", b, int(s), 1, N, "cpu").numpy()))[0]
                for s in sel if s >= 0}
        o_ref, lse_ref, _ = O.sparse_attn(wl["q"][b, 0].double().cpu().numpy(), rows, sel,
                                          wl["swa"][b].double().cpu().numpy(), 0, t,
                                          wl["sink"].double().cpu().numpy(), 128)
        assert_close(o.numpy(), o_ref, 2e-2, f"b{b}: merged attention vs oracle")
        assert_close(lse.numpy(), lse_ref, 2e-3, f"b{b}: merged lse vs oracle")
