"""The allocation-free attention entry point (for callers that may not allocate
device memory, so cannot pass a workspace) must give the same result as the
regular entry point with a full workspace.  Decode-sized shapes are used so the
keys really are split and the library's fixed device array is used; two calls in
a row with different inputs check that a call does not depend on what the
previous one left in that array.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, B=8, N=20000, H=64):
    q = W.normal_tensor((B, 1, H, 512), seed, 1, torch.bfloat16, DEV)
    kv = C.csa2_fp4_pack(W.normal_tensor((B, N, 512), seed, 2, torch.float32, DEV))
    swa = W.normal_tensor((B, 128, 512), seed, 3, torch.bfloat16, DEV)
    idx = torch.stack([W.distinct_sample(N - 1, 512, seed, b, DEV) for b in range(B)]).to(torch.int32)
    idx = idx.view(B, 1, 512).contiguous()
    q_pos = torch.full((B, 1), N - 1, dtype=torch.int64, device=DEV)
    sink = W.normal_tensor((H,), seed, 4, torch.float32, DEV)
    return q, kv, idx, swa, q_pos, sink


def test_noalloc_matches_regular_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    C.load()
    B, H = 8, 64
    assert C.csa2_sparse_attn_workspace_bytes(B, 1, H, 512, 128) > 0      # the key split is in use
    for seed in (9101, 9102):
        q, kv, idx, swa, q_pos, sink = _inputs(seed)
        ref, ref_lse = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, out_dtype=torch.float32, want_lse=True)
        out = torch.empty((B, 1, H, 512), dtype=torch.float32, device=DEV)
        lse = torch.empty((B, 1, H), dtype=torch.float32, device=DEV)
        C.csa2_sparse_attn_noalloc(q, kv, idx, swa, q_pos, out, sink, lse=lse)
        C.csa2_ctx_check()
        assert_close(to_np(out), to_np(ref), 2e-2, f"noalloc output, call {seed}")
        assert_close(to_np(lse), to_np(ref_lse), 1e-5, f"noalloc lse, call {seed}")
