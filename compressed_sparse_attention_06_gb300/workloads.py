"""Seeded synthetic inputs for the CSA2 hot path (the five workloads it is measured on).

This module only draws numbers. It holds none of the method's arithmetic: no
compression, no scoring, no selection, no attention and no FP4 packing. The CUDA
path and the CPU oracle both consume the tensors it returns; neither side's code
is used here.

Generator (counter based, so any sub-range can be drawn on its own and the same
recipe runs on CPU and GPU):

  * key(seed, stream)  = splitmix64(seed * 2^32 + stream)                 (host int)
  * r_i                = splitmix64(key + i)        (64-bit wrapping, element i)
  * u_i                = ((r_i >> 11) + 0.5) * 2^-53          in the open (0, 1)
  * normal element i   = sqrt(-2 ln u_{2i}) * cos(2 pi u_{2i+1})   (Box-Muller, f64)
  * the f64 value is then rounded to the storage dtype by torch.

Seeds follow ``seed = workload_id * 1000 + stream``; every tensor has its own
stream and each sequence of a batch is a distinct element range, so all
sequences differ.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

_MASK64 = (1 << 64) - 1


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit constant as a signed int64 (torch scalar)."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MUL1 = _s64(0xBF58476D1CE4E5B9)
_MUL2 = _s64(0x94D049BB133111EB)


def _splitmix64_int(x: int) -> int:
    """splitmix64 on a Python int (used for the per-stream key)."""
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & _MASK64
    return x ^ (x >> 31)


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor (torch's >> is arithmetic)."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _splitmix64(x: torch.Tensor) -> torch.Tensor:
    x = x + _GOLDEN
    x = (x ^ _srl(x, 30)) * _MUL1
    x = (x ^ _srl(x, 27)) * _MUL2
    return x ^ _srl(x, 31)


def stream_key(seed: int, stream: int) -> int:
    return _s64(_splitmix64_int(((seed & 0xFFFFFFFF) << 32) | (stream & 0xFFFFFFFF)))


def uniform(count: int, seed: int, stream: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """f64 uniforms in (0, 1) for elements [offset, offset + count)."""
    key = stream_key(seed, stream)
    idx = torch.arange(offset, offset + count, dtype=torch.int64, device=device)
    r = _splitmix64(idx + key)
    return (_srl(r, 11).to(torch.float64) + 0.5) * (2.0 ** -53)


_CHUNK = 1 << 24


def normal(count: int, seed: int, stream: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """f64 standard normals for elements [offset, offset + count) of a stream."""
    out = torch.empty(count, dtype=torch.float64, device=device)
    key = stream_key(seed, stream)
    two_pi = 2.0 * math.pi
    for c0 in range(0, count, _CHUNK):
        n = min(_CHUNK, count - c0)
        i = torch.arange(offset + c0, offset + c0 + n, dtype=torch.int64, device=device)
        r1 = _splitmix64(2 * i + key)
        r2 = _splitmix64(2 * i + 1 + key)
        u1 = (_srl(r1, 11).to(torch.float64) + 0.5) * (2.0 ** -53)
        u2 = (_srl(r2, 11).to(torch.float64) + 0.5) * (2.0 ** -53)
        out[c0:c0 + n] = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(two_pi * u2)
    return out


def normal_tensor(shape, seed: int, stream: int, dtype=torch.float32, device="cpu",
                  std: float = 1.0, offset: int = 0) -> torch.Tensor:
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=dtype, device=device)
    for c0 in range(0, n, _CHUNK):
        k = min(_CHUNK, n - c0)
        out[c0:c0 + k] = (normal(k, seed, stream, device, offset + c0) * std).to(dtype)
    return out.view(*shape)


def distinct_sample(population: int, k: int, seed: int, stream: int, device="cpu") -> torch.Tensor:
    """k distinct integers drawn uniformly from [0, population), ascending (int64).

    Each candidate gets a uniform key; the k smallest keys win (a seeded
    partial shuffle)."""
    if k > population:
        raise ValueError("k > population")
    u = uniform(population, seed, stream, device)
    sel = torch.topk(u, k, largest=False).indices
    return torch.sort(sel).values


def snap(x: torch.Tensor, step: float, lim: float) -> torch.Tensor:
    """Round values to the nearest multiple of `step` and clip them to [-lim, lim]:
    the exact-grid variant of a workload (every product and partial sum of the
    indexer is then exact in fp32, so scores and selections must match bit for bit)."""
    return torch.clamp(torch.round(x.double() / step) * step, -lim, lim)


# Exact-grid FP4 rows: values from this signed set, with the first value of every
# 32-value block set to 4, so each block's largest magnitude is 4 and its MXFP4
# scale is 2^0: every value is then stored exactly.
_FP4_GRID = (-4.0, -3.0, -2.0, -1.5, -1.0, -0.5, 0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0)


def fp4_grid_rows(seed: int, stream: int, row0: int, rows: int, width: int, device="cpu") -> torch.Tensor:
    """[rows, width] f32 rows of the exact-grid FP4 workload (rows row0 .. of a stream)."""
    u = uniform(rows * width, seed, stream, device, offset=row0 * width)
    vals = torch.tensor(_FP4_GRID, dtype=torch.float64, device=device)
    x = vals[torch.clamp((u * len(_FP4_GRID)).long(), max=len(_FP4_GRID) - 1)].view(rows, width // 32, 32)
    x[:, :, 0] = 4.0
    return x.reshape(rows, width).to(torch.float32)


# ----------------------------------------------------------------------------------
# The five workloads.  Shapes, dtypes and distributions are those of the workload
# descriptions; `scale` knobs shrink a workload for the fast tests while keeping
# its structure (same m, heads, dims, k, window and pool sizes).
# ----------------------------------------------------------------------------------

TOPK = 512
WINDOW = 128
POOL_BLOCK = 8
POOL_KEEP = 2048
C_MAIN = 512
D_INDEX = 128


@dataclass
class Workload:
    name: str
    B: int
    Q: int
    N: int                      # compressed entries per sequence in the cache
    m: int
    H_I: int
    H: int
    q_pos: torch.Tensor         # [B, Q] int64 query positions
    tensors: Dict[str, torch.Tensor] = field(default_factory=dict)
    meta: Dict[str, object] = field(default_factory=dict)

    def __getitem__(self, k):
        return self.tensors[k]


def _wid_seed(wid: int, stream: int) -> int:
    return wid * 1000 + stream


def tiny_full_layer(device="cpu") -> Workload:
    """Tiny CSA2 Full layer, fp32: n=4096 tokens, c=512, m=2 (no overlap, B^a=0) ->
    2048 entries; indexer K 2048x128; 8 indexer heads; 16 core heads; four decode
    queries at positions 4095..4092; 128-token window; sink 0."""
    wid = 1
    n, c, m = 4096, C_MAIN, 2
    N = n // m
    B, Q, H_I, H = 1, 4, 8, 16
    t = {}
    t["Ca"] = normal_tensor((n, c), _wid_seed(wid, 1), 0, torch.float32, device)
    t["Za"] = normal_tensor((n, c), _wid_seed(wid, 2), 0, torch.float32, device)
    t["Ba"] = torch.zeros((m, c), dtype=torch.float32, device=device)
    t["KI"] = normal_tensor((B, N, D_INDEX), _wid_seed(wid, 3), 0, torch.float32, device)
    t["qI"] = normal_tensor((B, Q, H_I, D_INDEX), _wid_seed(wid, 4), 0, torch.float32, device)
    t["w"] = normal_tensor((B, Q, H_I), _wid_seed(wid, 5), 0, torch.float32, device)
    t["q"] = normal_tensor((B, Q, H, c), _wid_seed(wid, 6), 0, torch.float32, device)
    t["swa"] = normal_tensor((B, n, c), _wid_seed(wid, 7), 0, torch.float32, device)
    t["sink"] = torch.zeros(H, dtype=torch.float32, device=device)
    q_pos = torch.tensor([[4095, 4094, 4093, 4092]], dtype=torch.int64, device=device)
    return Workload("tiny_full_layer_fp32", B, Q, N, m, H_I, H, q_pos, t,
                    dict(n_tokens=n, swa_pos0=0, swa_cap=n, pos0=0, dtype="f32"))


def plant_direction(qI: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    """Unit direction d/|d| with d = sum_h max(w_h, 0) q^I_h, per query (f64).

    qI: [..., H_I, d], w: [..., H_I] -> [..., d].  A key placed along this
    direction lines up with the positively weighted indexer heads."""
    d = (w.double().clamp_min(0.0).unsqueeze(-1) * qI.double()).sum(-2)
    return d / d.norm(dim=-1, keepdim=True).clamp_min(1e-300)


# Planted-key length: the smallest multiple of 0.25 at or above 12 * sqrt(128),
# about twelve times the length of a random N(0,1) key of 128 dims.
PLANT_BETA = math.ceil(12.0 * math.sqrt(D_INDEX) * 4.0) / 4.0
N_PLANTED = 16


def decode_full_bf16(device="cpu", B: int = 32, N: int = 65536, with_main_kv: bool = True,
                     grid: bool = False) -> Workload:
    """Decoder Full-mode decode, bf16: B sequences, N entries (m=1), query at
    t = N-1 (V = N-1), 64 indexer heads, 64 core heads, 16 planted keys per
    sequence at seeded positions in [0, V-129), 128-token window ring, sink 0.

    grid=True: the exact-grid variant -- q^I and K^I on multiples of 2^-3 in
    [-4, 4], w on multiples of 2^-1 in [-4, 4], no planted keys (they are off grid)."""
    wid = 2
    m, H_I, H, Q = 1, 64, 64, 1
    t = {}
    if with_main_kv:
        t["kv"] = normal_tensor((B, N, C_MAIN), _wid_seed(wid, 1), 0, torch.bfloat16, device)
    KI = normal_tensor((B, N, D_INDEX), _wid_seed(wid, 2), 0, torch.bfloat16, device)
    t["qI"] = normal_tensor((B, Q, H_I, D_INDEX), _wid_seed(wid, 3), 0, torch.bfloat16, device)
    t["w"] = normal_tensor((B, Q, H_I), _wid_seed(wid, 4), 0, torch.float32, device)
    if grid:
        KI = snap(KI, 0.125, 4.0).to(torch.bfloat16)
        t["qI"] = snap(t["qI"], 0.125, 4.0).to(torch.bfloat16)
        t["w"] = snap(t["w"], 0.5, 4.0).to(torch.float32)
    t["q"] = normal_tensor((B, Q, H, C_MAIN), _wid_seed(wid, 5), 0, torch.bfloat16, device)
    t["swa"] = normal_tensor((B, WINDOW, C_MAIN), _wid_seed(wid, 6), 0, torch.bfloat16, device)
    t["sink"] = torch.zeros(H, dtype=torch.float32, device=device)
    V = N - 1
    span = max(V - 129, 1)
    planted = torch.empty((B, N_PLANTED), dtype=torch.int64, device=device)
    u_dir = plant_direction(t["qI"][:, 0], t["w"][:, 0])            # [B, 128]
    for b in range(0 if grid else B):
        pos = distinct_sample(span, min(N_PLANTED, span), _wid_seed(wid, 7) + 17 * b, b, device)
        planted[b, :pos.numel()] = pos
        KI[b, pos] = (PLANT_BETA * u_dir[b]).to(torch.bfloat16).unsqueeze(0).expand(pos.numel(), -1)
    t["KI"] = KI
    if not grid:
        t["planted"] = planted
    # the new token's compressor inputs (m = 1: one row) and its indexer key row
    t["C_new"] = normal_tensor((B, 1, C_MAIN), _wid_seed(wid, 8), 0, torch.bfloat16, device)
    t["Z_new"] = normal_tensor((B, 1, C_MAIN), _wid_seed(wid, 9), 0, torch.bfloat16, device)
    t["KI_new"] = normal_tensor((B, 1, D_INDEX), _wid_seed(wid, 10), 0, torch.bfloat16, device)
    q_pos = torch.full((B, Q), N - 1, dtype=torch.int64, device=device)
    return Workload("decode_full_bf16" + ("_grid" if grid else ""), B, Q, N, m, H_I, H, q_pos, t,
                    dict(swa_pos0=0, swa_cap=WINDOW, dtype="bf16"))


def reindex_reuse_bf16(device="cpu", B: int = 64, N: int = 262144, n_reuse: int = 3,
                       with_main_kv: bool = True, grid: bool = False) -> Workload:
    """Reindex + Reuse decode, bf16: each query rescores its 2048 pooled blocks
    (16,384 candidates) with its own indexer q/w, takes top-512, then the Reindex
    layer and three Reuse layers each attend with their own q and window.

    grid=True: the exact-grid variant (q^I, K^I on multiples of 2^-3 in [-4, 4],
    w on multiples of 2^-1 in [-4, 4])."""
    wid = 3
    m, H_I, H, Q = 1, 64, 64, 1
    t = {}
    if with_main_kv:
        t["kv"] = normal_tensor((B, N, C_MAIN), _wid_seed(wid, 1), 0, torch.bfloat16, device)
    t["KI"] = normal_tensor((B, N, D_INDEX), _wid_seed(wid, 2), 0, torch.bfloat16, device)
    t["qI"] = normal_tensor((B, Q, H_I, D_INDEX), _wid_seed(wid, 3), 0, torch.bfloat16, device)
    t["w"] = normal_tensor((B, Q, H_I), _wid_seed(wid, 4), 0, torch.float32, device)
    if grid:
        for nm in ("KI", "qI"):
            t[nm] = snap(t[nm], 0.125, 4.0).to(torch.bfloat16)
        t["w"] = snap(t["w"], 0.5, 4.0).to(torch.float32)
    V = N - 1
    b_new = (V - 1) // POOL_BLOCK
    n_keep = min(POOL_KEEP, b_new + 1)
    pool = torch.full((B, Q, POOL_KEEP), -1, dtype=torch.int32, device=device)
    for b in range(B):
        others = distinct_sample(b_new, n_keep - 1, _wid_seed(wid, 5) + 31 * b, b, device)
        blocks = torch.cat([others, torch.tensor([b_new], dtype=torch.int64, device=device)])
        pool[b, 0, :n_keep] = torch.sort(blocks).values.to(torch.int32)
    t["pool"] = pool
    for layer in range(1 + n_reuse):
        t[f"q{layer}"] = normal_tensor((B, Q, H, C_MAIN), _wid_seed(wid, 10 + layer), 0,
                                       torch.bfloat16, device)
        t[f"swa{layer}"] = normal_tensor((B, WINDOW, C_MAIN), _wid_seed(wid, 20 + layer), 0,
                                         torch.bfloat16, device)
    t["sink"] = torch.zeros(H, dtype=torch.float32, device=device)
    q_pos = torch.full((B, Q), N - 1, dtype=torch.int64, device=device)
    return Workload("reindex_reuse_bf16" + ("_grid" if grid else ""), B, Q, N, m, H_I, H, q_pos, t,
                    dict(swa_pos0=0, swa_cap=WINDOW, n_layers=1 + n_reuse, dtype="bf16"))


def fp4_rows(kind: str, b: int, row0: int, rows: int, N: int, device="cpu") -> torch.Tensor:
    """Float rows of the FP4-cache decode workload before packing, f32.

    kind 'kv' -> [rows, 512], kind 'KI' -> [rows, 128]; x ~ N(0,1) * r_row with
    r_row ~ LogNormal(0, 0.5) per row.  Rows [row0, row0+rows) of sequence b."""
    wid = 4
    width, s_val, s_row = (C_MAIN, 1, 2) if kind == "kv" else (D_INDEX, 3, 4)
    base_row = b * N + row0
    x = normal(rows * width, _wid_seed(wid, s_val), 0, device, offset=base_row * width)
    r = torch.exp(0.5 * normal(rows, _wid_seed(wid, s_row), 0, device, offset=base_row))
    return (x.view(rows, width) * r.view(rows, 1)).to(torch.float32)


def fp4_decode(device="cpu", B: int = 8, N: int = 1 << 20, H: int = 64, grid: bool = False) -> Workload:
    """FP4-cache long-context decode: B sequences of N entries (m=1); query at
    t = N-1.  The main-KV and indexer-K caches are drawn with `fp4_rows` and
    packed by the caller (FP4 E2M1+E4M3/16 and MXFP4 respectively).  H query heads
    (64; 128 for the V4-Pro configuration).

    grid=True: the exact-grid variant -- the indexer query from `fp4_grid_rows`
    (stored exactly by MXFP4), w on multiples of 2^-1 in [-4, 4]; the caller
    draws the indexer keys with `fp4_grid_rows` too."""
    wid = 4
    m, H_I, Q = 1, 64, 1
    t = {}
    t["qI"] = normal_tensor((B, Q, H_I, D_INDEX), _wid_seed(wid, 5), 0, torch.bfloat16, device)
    t["w"] = normal_tensor((B, Q, H_I), _wid_seed(wid, 6), 0, torch.float32, device)
    if grid:
        t["qI"] = fp4_grid_rows(_wid_seed(wid, 12), 0, 0, B * Q * H_I, D_INDEX, device).to(
            torch.bfloat16).view(B, Q, H_I, D_INDEX)
        t["w"] = snap(t["w"], 0.5, 4.0).to(torch.float32)
    t["q"] = normal_tensor((B, Q, H, C_MAIN), _wid_seed(wid, 7), 0, torch.bfloat16, device)
    t["swa"] = normal_tensor((B, WINDOW, C_MAIN), _wid_seed(wid, 8), 0, torch.bfloat16, device)
    t["sink"] = torch.zeros(H, dtype=torch.float32, device=device)
    t["C_new"] = normal_tensor((B, 1, C_MAIN), _wid_seed(wid, 9), 0, torch.bfloat16, device)
    t["Z_new"] = normal_tensor((B, 1, C_MAIN), _wid_seed(wid, 10), 0, torch.bfloat16, device)
    t["KI_new"] = normal_tensor((B, 1, D_INDEX), _wid_seed(wid, 11), 0, torch.bfloat16, device)
    q_pos = torch.full((B, Q), N - 1, dtype=torch.int64, device=device)
    return Workload("fp4_decode_1M", B, Q, N, m, H_I, H, q_pos, t,
                    dict(swa_pos0=0, swa_cap=WINDOW, dtype="fp4"))


def prefill_chunk_bf16(device="cpu", n_new: int = 8192, ctx_tokens: int = 131072,
                       q_stride: int = 1) -> Workload:
    """Encoder prefill chunk, bf16: B=1, n_new causal queries appended to a
    ctx_tokens context; overlapped compressor with m=4 (B^a, B^b ~ N(0, 0.1);
    previous-block state = the context's last m tokens' C^b/Z^b); 64 indexer heads,
    top-512, 64 core heads, 128 window, sink ~ N(0,1) per head.

    q_stride > 1 keeps every q_stride-th query only (for reduced tests)."""
    wid = 5
    m, H_I, H = 4, 64, 64
    n_ctx_entries = ctx_tokens // m
    N = (ctx_tokens + n_new) // m
    qpos_all = torch.arange(ctx_tokens, ctx_tokens + n_new, dtype=torch.int64, device=device)
    q_pos = qpos_all[::q_stride].reshape(1, -1)
    Q = q_pos.shape[1]
    t = {}
    t["kv_ctx"] = normal_tensor((1, n_ctx_entries, C_MAIN), _wid_seed(wid, 1), 0, torch.bfloat16, device)
    for i, nm in enumerate(["Ca", "Cb", "Za", "Zb"]):
        t[nm] = normal_tensor((n_new, C_MAIN), _wid_seed(wid, 2 + i), 0, torch.bfloat16, device)
    t["Ba"] = normal_tensor((m, C_MAIN), _wid_seed(wid, 6), 0, torch.float32, device, std=0.1)
    t["Bb"] = normal_tensor((m, C_MAIN), _wid_seed(wid, 7), 0, torch.float32, device, std=0.1)
    t["prev_Cb"] = normal_tensor((m, C_MAIN), _wid_seed(wid, 8), 0, torch.bfloat16, device)
    t["prev_Zb"] = normal_tensor((m, C_MAIN), _wid_seed(wid, 9), 0, torch.bfloat16, device)
    t["KI"] = normal_tensor((1, N, D_INDEX), _wid_seed(wid, 10), 0, torch.bfloat16, device)
    # per-query tensors are drawn for the full chunk and then strided, so a reduced
    # test sees exactly the rows the full workload has at those positions
    qI = normal_tensor((n_new, H_I, D_INDEX), _wid_seed(wid, 11), 0, torch.bfloat16, device)
    w = normal_tensor((n_new, H_I), _wid_seed(wid, 12), 0, torch.float32, device)
    q = normal_tensor((n_new, H, C_MAIN), _wid_seed(wid, 13), 0, torch.bfloat16, device)
    t["qI"] = qI[::q_stride].unsqueeze(0).contiguous()
    t["w"] = w[::q_stride].unsqueeze(0).contiguous()
    t["q"] = q[::q_stride].unsqueeze(0).contiguous()
    t["sink"] = normal_tensor((H,), _wid_seed(wid, 14), 0, torch.float32, device)
    swa_pos0 = max(0, ctx_tokens - WINDOW + 1)
    n_swa = ctx_tokens + n_new - swa_pos0
    t["swa"] = normal_tensor((1, n_swa, C_MAIN), _wid_seed(wid, 15), 0, torch.bfloat16, device)
    return Workload("prefill_chunk_bf16", 1, Q, N, m, H_I, H, q_pos, t,
                    dict(swa_pos0=swa_pos0, swa_cap=n_swa, pos0=ctx_tokens,
                         n_ctx_entries=n_ctx_entries, n_new=n_new, dtype="bf16"))
