"""HCA on the GPU (DSA-to-CSA/HCA page «HCA：公式 (20)–(26)»): the m' = 128
non-overlapping compressor against the oracle, and csa2_dense_attn -- every visible
compressed entry plus the window -- against the oracle on both attention paths
(tensor cores: bf16 query and window, bf16 or FP4 rows, both norms; CUDA cores: f32),
at small and at 1M-context sizes, and bit-exact against csa2_sparse_attn given the
full index list."""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_06_gb300 import csa2 as C
from compressed_sparse_attention_06_gb300 import workloads as W
from oracle import csa2_oracle as O
from tests.helpers import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
M_HCA = 128


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_compress_m128_against_oracle(dt):
    B, n = 2, M_HCA * 6
    ca = W.normal_tensor((B, n, 512), 501, 1, torch.float32, DEV).to(dt)
    za = W.normal_tensor((B, n, 512), 501, 2, torch.float32, DEV).to(dt)
    ba = W.normal_tensor((M_HCA, 512), 501, 3, torch.float32, DEV, std=0.1)
    out = C.csa2_compress(ca, za, M_HCA, ba=ba, flags=C.W_NORM | C.W_ROPE, out_fmt="f32")
    C.csa2_ctx_check()
    for b in range(B):
        E = O.compress(ca[b].double().cpu().numpy(), za[b].double().cpu().numpy(), M_HCA,
                       ba.double().cpu().numpy())
        ref = O.compress_write(E, O.NORM_W | O.ROPE_W, M_HCA, 0)
        assert_close(to_np(out[b]), ref, 1e-4 if dt == torch.float32 else 2e-3, f"entries b{b}")


def _case(seed, B, N, kv_kind, q_dt, cap=128):
    kv_f = W.normal_tensor((B, N, 512), seed, 1, torch.float32, DEV) * 1.2
    if kv_kind == "fp4":
        kv = C.csa2_fp4_pack(kv_f)
        kv_np = O.nvfp4_unpack(O.nvfp4_pack(kv_f.reshape(-1, 512).cpu().numpy())).reshape(B, N, 512)
    else:
        kv = kv_f.to(q_dt)
        kv_np = kv.double().cpu().numpy()
    swa = W.normal_tensor((B, cap, 512), seed, 2, torch.float32, DEV).to(q_dt)
    sink = W.normal_tensor((128,), seed, 3, torch.float32, DEV)
    return kv, kv_np, swa, sink


def _check(q, kv_np, swa, sink, q_pos, out, lse, pairs, H, tol):
    for b, qq in pairs:
        t = int(q_pos[b, qq])
        o, l, _ = O.dense_attn(q[b, qq].double().cpu().numpy(), kv_np[b], swa[b].double().cpu().numpy(), 0, t,
                               M_HCA, sink[:H].double().cpu().numpy(), 128)
        assert_close(to_np(out[b, qq].float()), o, tol, f"out b{b} q{qq} t{t}")
        assert_close(to_np(lse[b, qq]), l, 2e-3 if tol > 1e-3 else 1e-5, f"lse b{b} q{qq}")


@pytest.mark.parametrize("kv_kind,q_dt,H", [("bf16", torch.bfloat16, 64), ("fp4", torch.bfloat16, 64),
                                            ("f32", torch.float32, 16), ("bf16", torch.bfloat16, 96)])
def test_dense_attn_small(kv_kind, q_dt, H):
    """V from 0 to 40 entries (t from 100 to 5,200), ragged tiles, both paths (H = 96
    and f32 take the CUDA cores)."""
    B, Q, N = 2, 3, 48
    kv, kv_np, swa, sink = _case(511, B, N, kv_kind, q_dt)
    q = W.normal_tensor((B, Q, H, 512), 512, 1, torch.float32, DEV).to(q_dt)
    q_pos = torch.tensor([[100, 1000, 40 * M_HCA + 5], [M_HCA, M_HCA * 17 - 1, M_HCA * 33]], dtype=torch.int64,
                         device=DEV)
    nv = torch.div(q_pos, M_HCA, rounding_mode="floor")
    out, lse = C.csa2_dense_attn(q, kv, nv, N, swa, q_pos, sink[:H].contiguous(), window=128,
                                 out_dtype=torch.float32, want_lse=True)
    C.csa2_ctx_check()
    tol = 1e-4 if q_dt == torch.float32 else 2e-2
    _check(q, kv_np, swa, sink, q_pos, out, lse, [(b, qq) for b in range(B) for qq in range(Q)], H, tol)


def test_dense_attn_1M_context_fp4():
    """1M-token context: 8,192 HCA entries per sequence in FP4; queries near the end
    (V = 8,191) and mid-way; sampled through the oracle."""
    B, N = 2, 8192
    kv, kv_np, swa, sink = _case(521, B, N, "fp4", torch.bfloat16)
    q = W.normal_tensor((B, 1, 64, 512), 522, 1, torch.float32, DEV).to(torch.bfloat16)
    q_pos = torch.tensor([[(1 << 20) - 1], [300000]], dtype=torch.int64, device=DEV)
    nv = torch.div(q_pos, M_HCA, rounding_mode="floor")
    out, lse = C.csa2_dense_attn(q, kv, nv, N, swa, q_pos, sink[:64].contiguous(), window=128,
                                 out_dtype=torch.float32, want_lse=True)
    C.csa2_ctx_check()
    _check(q, kv_np, swa, sink, q_pos, out, lse, [(0, 0), (1, 0)], 64, 2e-2)


@pytest.mark.parametrize("kv_kind", ["bf16", "fp4"])
def test_dense_equals_sparse_with_every_index(kv_kind):
    """One query: the dense call over V entries and the sparse call with idx = 0..V-1
    (k = V) run the same slots through the same kernel: identical outputs."""
    N, V = 1500, 1500
    kv, _, swa, sink = _case(531, 1, N, kv_kind, torch.bfloat16)
    q = W.normal_tensor((1, 1, 64, 512), 532, 1, torch.float32, DEV).to(torch.bfloat16)
    q_pos = torch.tensor([[V * M_HCA + 3]], dtype=torch.int64, device=DEV)
    nv = torch.tensor([[V]], dtype=torch.int64, device=DEV)
    sink = sink[:64].contiguous()
    dense, dl = C.csa2_dense_attn(q, kv, nv, V, swa, q_pos, sink, window=128, out_dtype=torch.float32, want_lse=True)
    idx = torch.arange(V, dtype=torch.int32, device=DEV).view(1, 1, V)
    sparse, sl = C.csa2_sparse_attn(q, kv, idx, swa, q_pos, sink, window=128, out_dtype=torch.float32, want_lse=True)
    C.csa2_ctx_check()
    np.testing.assert_array_equal(to_np(dense), to_np(sparse))
    np.testing.assert_array_equal(to_np(dl), to_np(sl))
