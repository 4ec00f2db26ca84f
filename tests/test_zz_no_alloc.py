"""The allocation-free attention entry point must give the same result as the
regular entry point with a full workspace.

Some callers cannot allocate device memory (a serving engine that owns one arena
for the whole GPU and forbids cudaMalloc in plugins, or a latency-critical loop),
so they cannot pass a workspace; csa2_sparse_attn_noalloc keeps its partial
results in a fixed array inside the library instead.  Decode-sized shapes are used
so the keys really are split and that array is used; two calls in a row with
different inputs check that a call does not depend on what the previous one left
in the array.  Both kernel paths are covered: the tensor-core path (bf16 query,
FP4 rows, both norms) and the CUDA-core path (fp32 query), each bit for bit
against the regular entry point, since both calls run the same kernels with the
same key split.  This file is collected last on purpose."""
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, q_dtype, B=8, N=20000, H=64):
    q = W.normal_tensor((B, 1, H, 512), seed, 1, q_dtype, DEV)
    kv = C.csa2_fp4_pack(W.normal_tensor((B, N, 512), seed, 2, torch.float32, DEV))
    swa = W.normal_tensor((B, 128, 512), seed, 3, q_dtype, DEV)
    idx = torch.stack([W.distinct_sample(N - 1, 512, seed, b, DEV) for b in range(B)]).to(torch.int32)
    idx = idx.view(B, 1, 512).contiguous()
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=DEV)
    sink = W.normal_tensor((H,), seed, 4, torch.float32, DEV)
    return q, kv, idx, swa, q_pos, sink


@pytest.mark.parametrize("q_dtype", [torch.bfloat16, torch.float32], ids=["tensor_core", "cuda_core"])
def test_noalloc_matches_regular_entry_point_twice(q_dtype):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    B, H = 8, 64
    assert C.csa2_sparse_attn_workspace_bytes(B, 1, H, 512, 128) > 0      # the key split is in use
    for seed in (9101, 9102):
        q, kv, idx, swa, q_pos, sink = _inputs(seed, q_dtype)
        ref, ref_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, out_dtype=torch.float32, want_lse=True)
        # guarded buffers (in the GPU tests the binding's allocator adds guard bytes)
        out = C.alloc((B, 1, H, 512), dtype=torch.float32, device=DEV).fill_(float("nan"))
        lse = C.alloc((B, 1, H), dtype=torch.float32, device=DEV).fill_(float("nan"))
        C.csa2_sparse_attn_noalloc(q, kv, idx, swa, q_pos, out, sink, lse=lse)
        C.csa2_ctx_check()
        assert torch.equal(out, ref), f"noalloc output differs from csa2_sparse_attn, call {seed}"
        assert torch.equal(lse, ref_lse), f"noalloc lse differs from csa2_sparse_attn, call {seed}"


def test_noalloc_rejects_wrong_output_buffer():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    q, kv, idx, swa, q_pos, sink = _inputs(9103, torch.bfloat16, B=2, N=4096)
    small = torch.empty((2, 1, 32, 512), dtype=torch.float32, device=DEV)
    with pytest.raises(ValueError):
        C.csa2_sparse_attn_noalloc(q, kv, idx, swa, q_pos, small, sink)
    out = torch.empty((2, 1, 64, 512), dtype=torch.float32, device=DEV)
    with pytest.raises(ValueError):
        C.csa2_sparse_attn_noalloc(q, kv, idx, swa, q_pos, out, sink,
                                   lse=torch.empty((2, 1, 64), dtype=torch.bfloat16, device=DEV))
