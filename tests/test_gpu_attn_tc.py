"""Tensor-core sparse attention (bf16 query and window, bf16 or FP4 rows, both RMS
norms) against the oracle: single-split runs with many queries, key splits with
empty splits, ragged tiles, partial windows, padded idx, fewer than 64 heads, both
output dtypes; and against the CUDA-core path of the same call (no workspace)."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, B, Q, H, N, k, window, cap, pos, kv_kind, n_pad=0):
    q = W.normal_tensor((B, Q, H, 512), seed, 1, torch.bfloat16, DEV)
    kv_f = W.normal_tensor((B, N, 512), seed, 2, torch.float32, DEV) * 1.3
    if kv_kind == "fp4":
        kv = C.csa2_fp4_pack(kv_f)
        kv_np = O.nvfp4_unpack(O.nvfp4_pack(kv_f.reshape(-1, 512).cpu().numpy())).reshape(B, N, 512)
    else:
        kv = kv_f.to(torch.bfloat16)
        kv_np = kv.double().cpu().numpy()
    swa = W.normal_tensor((B, cap, 512), seed, 3, torch.bfloat16, DEV)
    q_pos = torch.tensor(pos, dtype=torch.int64, device=DEV).reshape(B, Q)
    idx = torch.full((B, Q, k), -1, dtype=torch.int32)
    for b in range(B):
        for qq in range(Q):
            n = k - (n_pad if (b + qq) % 2 else 0)
            idx[b, qq, :n] = W.distinct_sample(N, n, seed + 7 + b, qq).to(torch.int32)
    idx = idx.to(DEV)
    sink = W.normal_tensor((H,), seed, 4, torch.float32, DEV)
    return q, kv, kv_np, idx, swa, q_pos, sink


def _check(q, kv_np, idx, swa, q_pos, sink, window, out, lse, which, tol=2e-2):
    B, Q = q.shape[:2]
    for b, qq in which:
        o, l, _ = O.sparse_attn(q[b, qq].double().cpu().numpy(), kv_np[b], to_np(idx[b, qq]),
                                swa[b].double().cpu().numpy(), 0, int(q_pos[b, qq]),
                                sink.double().cpu().numpy(), window, C.ATTN_DEFAULT)
        assert_close(out[b, qq], o, tol, f"out b{b} q{qq}")
        assert_close(lse[b, qq], l, 2e-3, f"lse b{b} q{qq}")


@pytest.mark.parametrize("kv_kind", ["bf16", "fp4"])
def test_many_queries_single_split(kv_kind):
    """160 queries (one key split each), k = 300 (a ragged third tile), window 128."""
    B, Q, H, N, k, window = 1, 160, 64, 4000, 300, 128
    pos = [[N + 37 * i for i in range(Q)]]
    q, kv, kv_np, idx, swa, q_pos, sink = _case(301, B, Q, H, N, k, window, 128, pos, kv_kind, n_pad=41)
    assert C.csa2_sparse_attn_workspace_bytes(B, Q, H, k, window) >= B * Q * 65536
    out, lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                  want_lse=True)
    C.csa2_ctx_check()
    _check(q, kv_np, idx, swa, q_pos, sink, window, to_np(out), to_np(lse), [(0, i) for i in range(0, Q, 9)])


@pytest.mark.parametrize("kv_kind", ["bf16", "fp4"])
@pytest.mark.parametrize("out_dt", [torch.float32, torch.bfloat16])
def test_key_splits_with_empty_splits(kv_kind, out_dt):
    """Four queries, k = 200 and a 300-slot window (4 tiles, split 4 ways): the early
    positions fill fewer tiles, so some splits hold no slot at all."""
    B, Q, H, N, k, window, cap = 2, 2, 64, 2500, 200, 300, 320
    pos = [[10, 5000], [299, 0]]
    q, kv, kv_np, idx, swa, q_pos, sink = _case(302, B, Q, H, N, k, window, cap, pos, kv_kind, n_pad=57)
    out, lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=out_dt, want_lse=True)
    C.csa2_ctx_check()
    _check(q, kv_np, idx, swa, q_pos, sink, window, to_np(out.float()), to_np(lse),
           [(b, qq) for b in range(B) for qq in range(Q)])


@pytest.mark.parametrize("kv_kind", ["bf16", "fp4"])
def test_tensor_core_matches_cuda_core_path(kv_kind):
    """The same call without a workspace runs on the CUDA cores in fp32; the two
    agree to the bf16 rounding of the tensor-core path."""
    B, Q, H, N, k, window = 3, 2, 40, 3000, 512, 128
    pos = [[N, N + 900], [130, 4000], [64, 77]]
    q, kv, kv_np, idx, swa, q_pos, sink = _case(303, B, Q, H, N, k, window, 128, pos, kv_kind, n_pad=100)
    tc, tc_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                    want_lse=True)
    tiny = torch.empty(16, dtype=torch.uint8, device=DEV)
    cc, cc_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                    want_lse=True, ws=tiny)
    C.csa2_ctx_check()
    assert_close(to_np(tc), to_np(cc), 2e-2, "tensor-core vs CUDA-core output")
    assert_close(to_np(tc_lse), to_np(cc_lse), 2e-3, "tensor-core vs CUDA-core lse")
    _check(q, kv_np, idx, swa, q_pos, sink, window, to_np(tc), to_np(tc_lse), [(0, 0), (2, 1)])


def test_tensor_core_out_of_range_index_is_flagged():
    B, Q, H, N = 1, 1, 64, 100
    q = torch.randn((B, Q, H, 512), device=DEV).to(torch.bfloat16)
    kv = torch.randn((B, N, 512), device=DEV).to(torch.bfloat16)
    swa = torch.randn((B, 128, 512), device=DEV).to(torch.bfloat16)
    idx = torch.tensor([[[3, 7, N + 5, -1]]], dtype=torch.int32, device=DEV)
    pos = torch.tensor([[50]], dtype=torch.int64, device=DEV)
    out, _ = C.csa2_sparse_attn(q, kv, idx, swa, pos, None, window=128)
    with pytest.raises(C.Csa2Error) as e:
        C.csa2_ctx_check()
    assert e.value.status == C.ERR_DEVICE
    C.csa2_ctx_check()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("H,k", [(128, 1024), (100, 512)])
@pytest.mark.parametrize("kv_kind", ["bf16", "fp4"])
def test_more_than_64_heads_in_passes(H, k, kv_kind):
    """More than 64 heads (V4-Pro: 128): the tensor-core path runs 64-head passes over
    the same rows (the second one ragged for H = 100), all in one launch, or one after
    another when the workspace holds one pass only; against the oracle, against each
    other and against the CUDA-core path of the same call."""
    B, Q, N, window = 2, 2, 6000, 128
    pos = [[N, N + 300], [700, 5000]]
    q = W.normal_tensor((B, Q, H, 512), 341, 1, torch.bfloat16, DEV)
    kv_f = W.normal_tensor((B, N, 512), 341, 2, torch.float32, DEV) * 1.3
    if kv_kind == "fp4":
        kv = C.csa2_fp4_pack(kv_f)
        kv_np = O.nvfp4_unpack(O.nvfp4_pack(kv_f.reshape(-1, 512).cpu().numpy())).reshape(B, N, 512)
    else:
        kv = kv_f.to(torch.bfloat16)
        kv_np = kv.double().cpu().numpy()
    swa = W.normal_tensor((B, 128, 512), 341, 3, torch.bfloat16, DEV)
    q_pos = torch.tensor(pos, dtype=torch.int64, device=DEV)
    idx = torch.full((B, Q, k), -1, dtype=torch.int32)
    for b in range(B):
        for qq in range(Q):
            n = k - (37 if (b + qq) % 2 else 0)
            idx[b, qq, :n] = W.distinct_sample(N, n, 342 + b, qq).to(torch.int32)
    idx = idx.to(DEV)
    sink = W.normal_tensor((H,), 343, 0, torch.float32, DEV)
    tc, tc_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                    want_lse=True)
    tiny = torch.empty(16, dtype=torch.uint8, device=DEV)
    cc, cc_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                    want_lse=True, ws=tiny)
    # a workspace below what all passes in one launch need: the passes run one after
    # another (or, below one pass's need, on the CUDA cores)
    full = C.csa2_sparse_attn_workspace_bytes(B, Q, H, k, window)
    one = torch.empty(max(16, min(C.csa2_sparse_attn_workspace_bytes(B, Q, 64, k, window), full - 1)),
                      dtype=torch.uint8, device=DEV)
    pp, pp_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                    want_lse=True, ws=one)
    C.csa2_ctx_check()
    assert_close(to_np(tc), to_np(cc), 2e-2, "tensor-core vs CUDA-core output")
    assert_close(to_np(tc_lse), to_np(cc_lse), 2e-3, "tensor-core vs CUDA-core lse")
    assert_close(to_np(tc), to_np(pp), 2e-2, "all passes in one launch vs the smaller workspace")
    assert_close(to_np(tc_lse), to_np(pp_lse), 2e-3, "all passes in one launch vs the smaller workspace (lse)")
    _check(q, kv_np, idx, swa, q_pos, sink, window, to_np(tc), to_np(tc_lse), [(0, 1), (1, 0)])
    _check(q, kv_np, idx, swa, q_pos, sink, window, to_np(pp), to_np(pp_lse), [(0, 0), (1, 1)])


@pytest.mark.parametrize("B", [8, 200])
def test_prepared_query_half_equals_one_call(B):
    """csa2_attn_prepare on another stream, then csa2_sparse_attn with ATTN_PREPARED on
    the same workspace, gives the one-call result bit for bit: decode shapes (a query's
    key splits merged in one cluster) and many queries (persistent CTAs)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    N, H = 20000, 64
    q = W.normal_tensor((B, 1, H, 512), 7301, 0, torch.bfloat16, DEV)
    kv = C.csa2_fp4_pack(W.normal_tensor((B, N, 512), 7302, 0, torch.float32, DEV))
    swa = W.normal_tensor((B, 128, 512), 7303, 0, torch.bfloat16, DEV)
    idx = torch.stack([W.distinct_sample(N - 1, 512, 7304, b, DEV) for b in range(B)]).to(torch.int32).view(B, 1, 512)
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=DEV)
    sink = W.normal_tensor((H,), 7305, 0, torch.float32, DEV)
    ref, ref_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, out_dtype=torch.float32, want_lse=True)
    ws = torch.empty(C.csa2_sparse_attn_workspace_bytes(B, 1, H, 512, 128, N=N, swa_cap=128), dtype=torch.uint8,
                     device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        C.csa2_attn_prepare(q, q_pos, ws, 512, window=128, N=N, swa_cap=128)
    torch.cuda.current_stream().wait_stream(side)
    out, lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, out_dtype=torch.float32, want_lse=True, ws=ws,
                                  flags=C.ATTN_DEFAULT | C.ATTN_PREPARED)
    C.csa2_ctx_check()
    assert torch.equal(out, ref)
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("shape", ["one_split", "key_splits"])
def test_bounded_wait_times_out_and_context_recovers(shape):
    """The attention kernel with a query-image producer that never signals (test
    hook): its consumers' bounded waits expire (about 2^27 cycles), the call reports
    a timeout instead of hanging, and the next call on the same context returns the
    same bits as a call made before the stall.  key_splits runs the splits of a
    query as one thread-block cluster (merged in the kernel)."""
    if shape == "one_split":
        B, Q, H, N, k, window, cap = 1, 4, 64, 3000, 300, 128, 128
        pos = [[N + 5 * i for i in range(Q)]]
    else:
        B, Q, H, N, k, window, cap = 2, 2, 64, 2500, 200, 300, 320
        pos = [[10, 5000], [299, 4000]]
    q, kv, kv_np, idx, swa, q_pos, sink = _case(311, B, Q, H, N, k, window, cap, pos, "fp4", n_pad=13)
    ref, ref_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                      want_lse=True)
    C.csa2_ctx_check()
    C.csa2_ctx_test_stall_next(1 << 27)
    C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32, want_lse=True)
    with pytest.raises(C.Csa2Error) as e:
        C.csa2_ctx_check()
    assert e.value.status == C.ERR_TIMEOUT
    out, lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=window, out_dtype=torch.float32,
                                  want_lse=True)
    C.csa2_ctx_check()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    _check(q, kv_np, idx, swa, q_pos, sink, window, to_np(out), to_np(lse), [(0, 0), (B - 1, Q - 1)])
