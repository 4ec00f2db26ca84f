"""Packed samples (varlen batches): compression windows, the window and the indexer's
visible range must not cross samples (DSA-to-CSA/HCA page, the note under the
compressor code and «算法语义»).  The varlen compressor writes each sample's entries
into the sample's own cache row, so the indexer, selection and attention -- run with
one row per sample -- stay inside the sample by construction; a padded query slot
(position -1) sees nothing."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import pipeline as P
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np, topk_swaps

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [37, 128, 5, 64, 0, 91, 3]


def _packed(seed, lens, c, dt, overlap=True):
    T = sum(lens)
    rows = [W.normal_tensor((T, c), seed, k, torch.float32, DEV).to(dt) for k in range(4)]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64, device=DEV)
    return rows[0], rows[1], (rows[2] if overlap else None), (rows[3] if overlap else None), cu


@pytest.mark.parametrize("fmt,c,dt", [("f32", 512, torch.float32), ("fp4", 512, torch.bfloat16),
                                      ("mxfp4", 128, torch.bfloat16), ("bf16", 512, torch.bfloat16)])
@pytest.mark.parametrize("overlap,m", [(True, 4), (False, 4), (True, 32)])
def test_varlen_equals_each_sample_alone(fmt, c, dt, overlap, m):
    """m = 32 splits each entry's rows over several row groups of the CTA."""
    ca, za, cb, zb, cu = _packed(601, LENS, c, dt, overlap)
    ba = W.normal_tensor((m, c), 602, 1, torch.float32, DEV, std=0.1)
    bb = W.normal_tensor((m, c), 602, 2, torch.float32, DEV, std=0.1) if overlap else None
    pos0 = torch.tensor([0, 400, 8, 1000, 0, 12, 4], dtype=torch.int64, device=DEV)
    flags = C.W_NORM | C.W_ROPE
    S, mx = len(LENS), max(LENS)
    out = C.csa2_compress_varlen(ca, za, m, cu, mx, cb=cb, zb=zb, ba=ba, bb=bb, pos0=pos0, flags=flags, out_fmt=fmt)
    C.csa2_ctx_check()
    for s_, n in enumerate(LENS):
        k = (n // m) * m
        if k == 0:
            continue
        a, b = int(cu[s_]), int(cu[s_]) + k
        sl = lambda t: None if t is None else t[a:b].contiguous()
        alone = C.csa2_compress(sl(ca), sl(za), m, cb=sl(cb), zb=sl(zb), ba=ba, bb=bb, pos0=int(pos0[s_]),
                                flags=flags, out_fmt=fmt)
        np.testing.assert_array_equal(to_np(out[s_, : n // m]), to_np(alone), err_msg=f"sample {s_}")
        if fmt == "f32":
            f = lambda t: None if t is None else t[a:b].double().cpu().numpy()
            E = O.compress(f(ca), f(za), m, ba.double().cpu().numpy(), f(cb), f(zb),
                           None if bb is None else bb.double().cpu().numpy())
            ref = O.compress_write(E, O.NORM_W | O.ROPE_W, m, int(pos0[s_]))
            assert_close(to_np(out[s_, : n // m]), ref, 1e-4, f"oracle sample {s_}")


def test_no_window_crosses_a_sample():
    """Changing every token of one sample changes no entry of any other sample, and a
    tail shorter than m (sample 2: 5 tokens = one block + 1) is not completed by the
    next sample's tokens."""
    m, c = 4, 512
    ca, za, cb, zb, cu = _packed(611, LENS, c, torch.float32)
    S, mx = len(LENS), max(LENS)
    base = C.csa2_compress_varlen(ca, za, m, cu, mx, cb=cb, zb=zb, out_fmt="f32")
    for s_ in range(S):
        a, b = int(cu[s_]), int(cu[s_ + 1])
        if a == b:
            continue
        ca2, za2, cb2, zb2 = ca.clone(), za.clone(), cb.clone(), zb.clone()
        for t in (ca2, za2, cb2, zb2):
            t[a:b] = torch.randn((b - a, c), device=DEV)
        out = C.csa2_compress_varlen(ca2, za2, m, cu, mx, cb=cb2, zb=zb2, out_fmt="f32")
        for o in range(S):
            ne = LENS[o] // m
            same = torch.equal(out[o, :ne], base[o, :ne])
            assert same == (o != s_ or ne == 0), (s_, o)
    C.csa2_ctx_check()


def test_packed_prefill_matches_samples_alone():
    """A varlen prefill batch as one row per sample (unequal numbers of valid entries,
    padded query slots at position -1): the top-k of each query equals that of its
    sample run alone, selection and attention agree with the oracle on the sample's
    own rows (attention is compared on the oracle's indices), and padded slots select
    nothing."""
    m, S, Qmax = 4, 3, 4
    lens = [4 * 300 + 2, 4 * 1000, 4 * 77 + 3]               # tokens per sample
    N = max(lens) // m
    ki = W.normal_tensor((S, N, 128), 621, 0, torch.float32, DEV).to(torch.bfloat16)
    kv = W.normal_tensor((S, N, 512), 622, 0, torch.float32, DEV).to(torch.bfloat16)
    swa = W.normal_tensor((S, max(lens), 512), 623, 0, torch.float32, DEV).to(torch.bfloat16)  # linear per sample
    pos = torch.full((S, Qmax), -1, dtype=torch.int64)
    for s_, n in enumerate(lens):
        for j in range(Qmax - (s_ == 2)):
            pos[s_, j] = n - 1 - 9 * j
    pos = pos.to(DEV)
    qI = W.normal_tensor((S, Qmax, 64, 128), 624, 0, torch.bfloat16, DEV)
    w = W.normal_tensor((S, Qmax, 64), 625, 0, torch.float32, DEV)
    q = W.normal_tensor((S, Qmax, 64, 512), 626, 0, torch.bfloat16, DEV)
    nv = P.visible_entries(pos, m)
    _, idx = P.full_topk_step(qI, w, ki, nv, k=512)
    C.csa2_ctx_check()
    for s_ in range(S):
        _, alone = P.full_topk_step(qI[s_:s_ + 1].contiguous(), w[s_:s_ + 1].contiguous(),
                                    ki[s_:s_ + 1].contiguous(), nv[s_:s_ + 1].contiguous(), k=512)
        np.testing.assert_array_equal(to_np(idx[s_]), to_np(alone[0]))
        for j in range(Qmax):
            t = int(pos[s_, j])
            if t < 0:
                assert torch.all(idx[s_, j] == -1)
                continue
            V = t // m
            sc = O.index_score(qI[s_, j].double().cpu().numpy(), w[s_, j].double().cpu().numpy(),
                               ki[s_].double().cpu().numpy(), V)
            topk_swaps(to_np(idx[s_, j]), sc, V, 512)
            ref_idx = O.topk(sc, V, 512)
            o, _, _ = O.sparse_attn(q[s_, j].double().cpu().numpy(), kv[s_].double().cpu().numpy(), ref_idx,
                                    swa[s_].double().cpu().numpy(), 0, t, None, 128)
            g, _ = C.csa2_sparse_attn(q[s_:s_ + 1, j:j + 1].contiguous(), kv[s_:s_ + 1].contiguous(),
                                      torch.tensor(ref_idx, dtype=torch.int32, device=DEV).view(1, 1, -1),
                                      swa[s_:s_ + 1].contiguous(), pos[s_:s_ + 1, j:j + 1].contiguous(), None,
                                      window=128, out_dtype=torch.float32)
            assert_close(to_np(g[0, 0]), o, 2e-2, f"attention sample {s_} query {j}")
    # the padded slots' attention is finite (the sink-free empty set gives zeros)
    out, _ = C.csa2_sparse_attn(q, kv, idx, swa, pos, None, window=128, out_dtype=torch.float32)
    C.csa2_ctx_check()
    assert torch.isfinite(out).all()
