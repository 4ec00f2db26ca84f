"""The decode compressor (csa2_compress_step) against the oracle and against the
whole-sequence kernel: streaming a sequence token by token, with the compressor
state of the Attention-evolution page §3.3, must produce exactly the entries of
compressing the whole sequence at once (DSA-to-CSA/HCA page eqs. (11)-(12); an
entry appears only when its block completes, «因果边界与短滑窗»)."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(B, n, c, seed, dt, overlap):
    ca = W.normal_tensor((B, n, c), seed, 1, torch.float32, DEV).to(dt)
    za = W.normal_tensor((B, n, c), seed, 2, torch.float32, DEV).to(dt)
    cb = W.normal_tensor((B, n, c), seed, 3, torch.float32, DEV).to(dt) if overlap else None
    zb = W.normal_tensor((B, n, c), seed, 4, torch.float32, DEV).to(dt) if overlap else None
    return ca, za, cb, zb


def _bias(m, c, seed, k):
    return W.normal_tensor((m, c), seed, k, torch.float32, DEV, std=0.1)


def _stream(ca, za, cb, zb, m, ba, bb, flags, out, fmt, start=0, state=None, skip=None):
    """Run positions start .. n-1 through csa2_compress_step; skip = {(b, p)} pairs
    that are sent as pos = -1 first and then again (the state must not change)."""
    B, n, c = ca.shape
    if state is None:
        state = C.csa2_compress_state(B, c, m, ca.dtype, DEV, overlap=cb is not None)
    for p in range(start, n):
        if skip:
            pos = torch.tensor([-1 if (b, p) in skip else p for b in range(B)], dtype=torch.int64, device=DEV)
            if (pos < 0).any():
                # a step where some sequences have no token: only the others advance
                C.csa2_compress_step(ca[:, p].contiguous(), za[:, p].contiguous(), m, pos, state,
                                     cb=None if cb is None else cb[:, p].contiguous(),
                                     zb=None if zb is None else zb[:, p].contiguous(), ba=ba, bb=bb, flags=flags,
                                     out=out, out_fmt=fmt, out_seq_stride=out.shape[1])
                pos = torch.tensor([p if (b, p) in skip else -1 for b in range(B)], dtype=torch.int64, device=DEV)
        else:
            pos = torch.full((B,), p, dtype=torch.int64, device=DEV)
        C.csa2_compress_step(ca[:, p].contiguous(), za[:, p].contiguous(), m, pos, state,
                             cb=None if cb is None else cb[:, p].contiguous(),
                             zb=None if zb is None else zb[:, p].contiguous(), ba=ba, bb=bb, flags=flags, out=out,
                             out_fmt=fmt, out_seq_stride=out.shape[1])
    return state


def _oracle_entries(ca, za, cb, zb, m, ba, bb, flags, b):
    f = lambda t: None if t is None else t[b].double().cpu().numpy()
    E = O.compress(f(ca), f(za), m, None if ba is None else ba.double().cpu().numpy(), f(cb), f(zb),
                   None if bb is None else bb.double().cpu().numpy())
    of = (O.NORM_W if flags & C.W_NORM else 0) | (O.ROPE_W if flags & C.W_ROPE else 0)
    return O.compress_write(E, of, m, 0)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("overlap,m", [(True, 4), (False, 2), (True, 1), (True, 16), (False, 128)])
def test_stream_equals_whole_sequence(dt, overlap, m):
    B, c = 3, 512
    n = 5 * m + (m - 1)                     # five complete blocks and an unfinished one
    ca, za, cb, zb = _rows(B, n, c, 401 + m, dt, overlap)
    ba, bb = _bias(m, c, 402, 1), (_bias(m, c, 402, 2) if overlap else None)
    flags = C.W_NORM | C.W_ROPE
    cap = n // m + 3
    out = torch.full((B, cap, c), 7.0, device=DEV)
    _stream(ca, za, cb, zb, m, ba, bb, flags, out, "f32")
    C.csa2_ctx_check()
    n_ent = n // m
    k = n_ent * m
    cut = lambda t: None if t is None else t[:, :k].contiguous()
    whole = C.csa2_compress(cut(ca), cut(za), m, cb=cut(cb), zb=cut(zb), ba=ba, bb=bb, flags=flags, out_fmt="f32")
    np.testing.assert_array_equal(to_np(out[:, :n_ent]), to_np(whole))          # same kernel math, bit-exact
    assert torch.all(out[:, n_ent:] == 7.0)                                     # the unfinished block wrote nothing
    for b in range(B):
        assert_close(to_np(out[b, :n_ent]), _oracle_entries(ca[:, : n_ent * m], za[:, : n_ent * m],
                                                            None if cb is None else cb[:, : n_ent * m],
                                                            None if zb is None else zb[:, : n_ent * m], m, ba, bb,
                                                            flags, b), 1e-4 if dt == torch.float32 else 2e-3,
                     f"entries b{b}")


@pytest.mark.parametrize("fmt,c,m", [("fp4", 512, 4), ("mxfp4", 128, 4), ("mxfp4", 128, 128)])
def test_stream_packed_cache_rows(fmt, c, m):
    """FP4 main-KV rows (c = 512) and MXFP4 indexer-key rows (c = 128) written straight
    into a cache: identical bytes to the whole-sequence kernel, and within the
    format's rounding of the oracle's entries (m = 128 with c = 128: sixteen row
    groups per entry)."""
    B = 2
    n = 6 * m
    ca, za, cb, zb = _rows(B, n, c, 411, torch.bfloat16, True)
    ba, bb = _bias(m, c, 412, 1), _bias(m, c, 412, 2)
    flags = C.W_NORM | (C.W_ROPE if c >= 128 else 0)
    rb = C.fp4_row_bytes(c) if fmt == "fp4" else C.mxfp4_row_bytes(c)
    cache = torch.zeros((B, 10, rb), dtype=torch.uint8, device=DEV)
    _stream(ca, za, cb, zb, m, ba, bb, flags, cache, fmt)
    C.csa2_ctx_check()
    whole = C.csa2_compress(ca, za, m, cb=cb, zb=zb, ba=ba, bb=bb, flags=flags, out_fmt=fmt)
    np.testing.assert_array_equal(to_np(cache[:, : n // m]), to_np(whole))
    for b in range(B):
        ref = _oracle_entries(ca, za, cb, zb, m, ba, bb, flags, b)
        if fmt == "fp4":
            got = O.nvfp4_unpack(to_np(cache[b, : n // m]), c)
            s = np.repeat(O.e4m3_decode(to_np(cache[b, : n // m, c // 2:])), 16, axis=1)
        else:
            got = O.mxfp4_unpack(to_np(cache[b, : n // m]), c)
            s = np.repeat(O.e8m0_decode(to_np(cache[b, : n // m, c // 2:])), 32, axis=1)
            # the oracle's own packing of its entry agrees to within one code step
        assert np.all(np.abs(got - ref) <= 2 * s + 1e-6), f"b{b}"


def test_skipped_steps_leave_the_state_alone():
    """Sequence 1 sits out some steps (pos = -1) and sends those tokens afterwards;
    the result equals the uninterrupted stream."""
    B, c, m = 3, 512, 4
    n = 4 * m
    ca, za, cb, zb = _rows(B, n, c, 421, torch.float32, True)
    ba, bb = _bias(m, c, 422, 1), _bias(m, c, 422, 2)
    out = torch.zeros((B, 6, c), device=DEV)
    _stream(ca, za, cb, zb, m, ba, bb, C.W_NORM, out, "f32", skip={(1, 3), (1, 7), (1, 8), (0, 12)})
    C.csa2_ctx_check()
    whole = C.csa2_compress(ca, za, m, cb=cb, zb=zb, ba=ba, bb=bb, flags=C.W_NORM, out_fmt="f32")
    np.testing.assert_array_equal(to_np(out[:, : n // m]), to_np(whole))


@pytest.mark.parametrize("n0", [0, 3, 8, 14])
def test_seeded_state_continues_a_prefix(n0):
    """A prefix of n0 tokens compressed with csa2_compress (carrying its last block
    into the next call), the state seeded from it, then the rest streamed: the
    entries equal compressing the whole sequence."""
    B, c, m = 2, 512, 4
    n = 22
    ca, za, cb, zb = _rows(B, n, c, 431 + n0, torch.bfloat16, True)
    ba, bb = _bias(m, c, 432, 1), _bias(m, c, 432, 2)
    flags = C.W_NORM | C.W_ROPE
    out = torch.zeros((B, 8, c), device=DEV)
    n0_full = (n0 // m) * m
    if n0_full:
        C.csa2_compress(ca[:, :n0_full].contiguous(), za[:, :n0_full].contiguous(), m,
                        cb=cb[:, :n0_full].contiguous(), zb=zb[:, :n0_full].contiguous(), ba=ba, bb=bb, flags=flags,
                        out=out, out_seq_stride=out.shape[1])
    state = C.csa2_compress_state(B, c, m, torch.bfloat16, DEV)
    C.csa2_compress_state_seed(ca[:, :n0].contiguous(), za[:, :n0].contiguous(), m, state,
                               cb=cb[:, :n0].contiguous(), zb=zb[:, :n0].contiguous())
    _stream(ca, za, cb, zb, m, ba, bb, flags, out, "f32", start=n0, state=state)
    C.csa2_ctx_check()
    whole = C.csa2_compress(ca[:, : (n // m) * m].contiguous(), za[:, : (n // m) * m].contiguous(), m,
                            cb=cb[:, : (n // m) * m].contiguous(), zb=zb[:, : (n // m) * m].contiguous(), ba=ba,
                            bb=bb, flags=flags, out_fmt="f32")
    np.testing.assert_array_equal(to_np(out[:, : n // m]), to_np(whole))
