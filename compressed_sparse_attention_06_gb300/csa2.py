"""Python binding of the CSA2 C ABI (libcsa2.so): argument marshalling only.

Each function has the name of its C entry point, takes torch CUDA tensors,
passes their data pointers and the current CUDA stream to the library, and
raises Csa2Error on a non-OK status.  Every step of the path runs in the
library's CUDA kernels; if the library is missing this module refuses to load.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa2.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(6)
F32, BF16, FP4_E4M3x16, MXFP4_E8M0x32 = range(4)
QNORM, KVNORM, ROPE = 1, 2, 4
ATTN_DEFAULT = QNORM | KVNORM | ROPE
ATTN_PREPARED = 8               # csa2_attn_prepare already wrote the query half into the workspace
W_NORM, W_ROPE = 1, 2
BLOCK_HIST_BINS = 4096          # words per row of csa2_index_score's block histogram

# symbols declared in include/csa2.h
EXPORTS = (
    "csa2_status_string", "csa2_version", "csa2_ctx_create", "csa2_ctx_destroy", "csa2_ctx_check",
    "csa2_ctx_test_stall_next",
    "csa2_compress", "csa2_fp4_pack", "csa2_fp4_unpack", "csa2_index_score", "csa2_topk",
    "csa2_block_pool", "csa2_sparse_attn", "csa2_sparse_attn_workspace_bytes", "csa2_sparse_attn_noalloc",
    "csa2_topk_workspace_bytes", "csa2_block_pool_workspace_bytes",
    "csa2_compress_step", "csa2_compress_state_bytes", "csa2_compress_state_seed", "csa2_dense_attn",
    "csa2_compress_varlen", "csa2_pool_topk", "csa2_block_hist", "csa2_attn_prepare", "csa2_visible_entries",
    "csa2_index_score_mxq",
)


class Csa2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_lib().csa2_status_string(status).decode()} (status {status})")


_LIB = None
_CTX = {}

_vp, _i, _i64, _u, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint, ctypes.c_float


def _declare(lib):
    sig = {
        "csa2_status_string": (ctypes.c_char_p, [_i]),
        "csa2_version": (_i, []),
        "csa2_ctx_create": (_i, [_i, ctypes.POINTER(_vp)]),
        "csa2_ctx_destroy": (_i, [_vp]),
        "csa2_ctx_check": (_i, [_vp, _vp]),
        "csa2_ctx_test_stall_next": (_i, [_vp, ctypes.c_longlong]),
        "csa2_compress": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i64, _i, _i, _vp, _f, _u,
                               _vp, _i, _i64, _vp]),
        "csa2_compress_step": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _f, _u, _vp, _i,
                                    _i64, _vp]),
        "csa2_compress_state_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i]),
        "csa2_compress_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _vp, _i64, _i, _i, _vp, _f, _u, _vp,
                                      _i, _i64, _vp]),
        "csa2_compress_state_seed": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _vp, _vp]),
        "csa2_fp4_pack": (_i, [_vp, _vp, _i, _i64, _i, _i, _vp, _i64, _vp]),
        "csa2_fp4_unpack": (_i, [_vp, _vp, _i, _i64, _i, _vp, _i, _vp]),
        "csa2_visible_entries": (_i, [_vp, _vp, _i64, _i, _vp, _vp]),
        "csa2_index_score_mxq": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp]),
        "csa2_index_score": (_i, [_vp, _vp, _i, _vp, _vp, _i, _i, _i, _i64, _i, _i, _vp, _vp, _i, _i, _vp,
                                  _vp, _vp, _vp]),
        "csa2_topk": (_i, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
        "csa2_topk_workspace_bytes": (ctypes.c_size_t, [_vp, _i64, _i64, _i]),
        "csa2_block_pool": (_i, [_vp, _vp, _vp, _i64, _i64, _vp, _i, _i, _vp, _vp, _i, _vp, ctypes.c_size_t,
                                 _vp]),
        "csa2_block_pool_workspace_bytes": (ctypes.c_size_t, [_vp, _i64, _i64, _i]),
        "csa2_attn_prepare": (_i, [_vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _i64, _i64, _f, _u, _vp,
                                   ctypes.c_size_t, _vp]),
        "csa2_block_hist": (_i, [_vp, _vp, _i64, _i64, _vp, _i, _vp, _vp]),
        "csa2_pool_topk": (_i, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _i, _i, _i, _vp, _vp, _vp, _vp]),
        "csa2_sparse_attn": (_i, [_vp, _vp, _i, _vp, _i, _i64, _vp, _i, _vp, _i, _i64, _i64, _i, _vp, _vp,
                                  _i, _i, _i, _i, _f, _u, _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]),
        "csa2_sparse_attn_workspace_bytes": (ctypes.c_size_t, [_vp, _i, _i, _i, _i, _i, _i64, _i64]),
        "csa2_dense_attn": (_i, [_vp, _vp, _i, _vp, _i, _i64, _vp, _i, _vp, _i, _i64, _i64, _i, _vp, _vp,
                                 _i, _i, _i, _i, _f, _u, _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]),
        "csa2_sparse_attn_noalloc": (_i, [_vp, _vp, _i, _vp, _i, _i64, _vp, _i, _vp, _i, _i64, _i64, _i, _vp, _vp,
                                          _i, _i, _i, _i, _f, _u, _vp, _i, _vp, _vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (the CSA2 path has no "
                              f"other implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        _declare(lib)
        _LIB = lib
    return _LIB


def load():
    """Load the library (raises if it is missing) and return the ctypes handle."""
    return _lib()


def ctx(device: Optional[int] = None):
    """The library context of a CUDA device (created on first use)."""
    if device is None:
        device = torch.cuda.current_device()
    if device not in _CTX:
        h = _vp()
        st = _lib().csa2_ctx_create(device, ctypes.byref(h))
        if st != OK:
            raise Csa2Error("csa2_ctx_create", st)
        _CTX[device] = h
    return _CTX[device]


def _stream(t: Optional[torch.Tensor] = None):
    dev = t.device if t is not None else torch.device("cuda", torch.cuda.current_device())
    return _vp(torch.cuda.current_stream(dev).cuda_stream)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("CSA2 tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("CSA2 tensors must be contiguous")
    return _vp(t.data_ptr())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def alloc(shape, dtype, device) -> torch.Tensor:
    """Every output and workspace this module (and pipeline.py) allocates comes from
    here: uninitialised device memory, like torch.empty.  The tests replace it with an
    allocator that puts guard bytes before and after each buffer."""
    return torch.empty(shape, dtype=dtype, device=device)


def _check(fn: str, st: int):
    if st != OK:
        raise Csa2Error(fn, st)


def fp4_row_bytes(c: int) -> int:
    return c // 2 + c // 16


def mxfp4_row_bytes(d: int) -> int:
    return d // 2 + d // 32


def csa2_ctx_check(device: Optional[int] = None):
    """Synchronise the current stream and raise if a kernel recorded an error."""
    dev = torch.cuda.current_device() if device is None else device
    _check("csa2_ctx_check", _lib().csa2_ctx_check(ctx(dev), _vp(torch.cuda.current_stream(dev).cuda_stream)))


def csa2_ctx_test_stall_next(budget_cycles: int = 0, device: Optional[int] = None):
    """Test hook: the next tensor-core indexer launch runs with a silent producer, so its
    bounded waits expire and csa2_ctx_check() raises a timeout."""
    _check("csa2_ctx_test_stall_next", _lib().csa2_ctx_test_stall_next(ctx(device), budget_cycles))


def csa2_fp4_pack(x: torch.Tensor, fmt: int = FP4_E4M3x16, out: Optional[torch.Tensor] = None,
                  out_ld: int = 0) -> torch.Tensor:
    """Pack rows [..., c] into FP4 (E2M1 + E4M3/16) or MXFP4 (E2M1 + E8M0/32) rows.
    With out_ld > 0, packed row r goes to byte offset r*out_ld of `out` (e.g. one new
    row per sequence written straight into a [B, N, row_bytes] cache)."""
    c = x.shape[-1]
    rows = x.numel() // c if c else 0
    rb = fp4_row_bytes(c) if fmt == FP4_E4M3x16 else mxfp4_row_bytes(c)
    if out is None:
        out = alloc((*x.shape[:-1], rb), dtype=torch.uint8, device=x.device)
        out_ld = 0
    ptr = _vp(out.data_ptr()) if out_ld else _p(out)
    _check("csa2_fp4_pack", _lib().csa2_fp4_pack(ctx(x.device.index), _p(x), _dt(x), rows, c, fmt, ptr, out_ld,
                                                 _stream(x)))
    return out


def csa2_fp4_unpack(b: torch.Tensor, fmt: int, c: int, out_dtype=torch.float32,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    rows = b.numel() // b.shape[-1] if b.shape[-1] else 0
    if out is None:
        out = alloc((*b.shape[:-1], c), dtype=out_dtype, device=b.device)
    _check("csa2_fp4_unpack", _lib().csa2_fp4_unpack(ctx(b.device.index), _p(b), fmt, rows, c, _p(out), _dt(out),
                                                     _stream(b)))
    return out


def _alloc_rows(shape, c, out_fmt, device):
    if out_fmt == "fp4":
        return alloc((*shape, fp4_row_bytes(c)), dtype=torch.uint8, device=device)
    if out_fmt == "mxfp4":
        return alloc((*shape, mxfp4_row_bytes(c)), dtype=torch.uint8, device=device)
    return alloc((*shape, c), dtype=torch.float32 if out_fmt == "f32" else torch.bfloat16, device=device)


def _out_dt(out, out_fmt):
    if out.dtype == torch.uint8:
        return MXFP4_E8M0x32 if out_fmt == "mxfp4" else FP4_E4M3x16
    return _dt(out)


def csa2_compress_varlen(ca, za, m: int, cu_tokens, max_tokens: int, cb=None, zb=None, ba=None, bb=None, pos0=None,
                         rope_base: float = 10000.0, flags: int = 0, out_fmt: str = "f32",
                         out: Optional[torch.Tensor] = None, out_seq_stride: Optional[int] = None):
    """Packed samples: ca/za (cb/zb) [T, c] hold S samples back to back, sample s at
    tokens cu_tokens[s] .. cu_tokens[s+1]-1 ([S+1] int64 device tensor).  Returns (or
    fills) [S, max_tokens // m, row]: entry i of sample s in row s, i; each sample is
    compressed alone (no shared window, tails left out)."""
    T, c = ca.shape
    S = cu_tokens.shape[0] - 1
    n_ent = max_tokens // m
    if out is None:
        out = _alloc_rows((S, n_ent), c, out_fmt, ca.device)
    oss = n_ent if out_seq_stride is None else out_seq_stride
    st = _lib().csa2_compress_varlen(ctx(ca.device.index), _p(ca), _p(za), _p(cb), _p(zb), _dt(ca), _p(ba), _p(bb), S,
                                     _p(cu_tokens), max_tokens, c, m, _p(pos0), rope_base, flags,
                                     _vp(out.data_ptr()), _out_dt(out, out_fmt), oss, _stream(ca))
    _check("csa2_compress_varlen", st)
    return out


def csa2_compress_state_bytes(B: int, c: int, m: int, dtype=torch.bfloat16, overlap: bool = True) -> int:
    return int(_lib().csa2_compress_state_bytes(B, c, m, F32 if dtype == torch.float32 else BF16, int(overlap)))


def csa2_compress_state(B: int, c: int, m: int, dtype, device, overlap: bool = True) -> torch.Tensor:
    """Device buffer for the decode compressor state (no clearing needed)."""
    return alloc(max(16, csa2_compress_state_bytes(B, c, m, dtype, overlap)), dtype=torch.uint8,
                       device=device)


def csa2_compress_step(ca, za, m: int, pos, state, cb=None, zb=None, ba=None, bb=None, rope_base: float = 10000.0,
                       flags: int = 0, out: Optional[torch.Tensor] = None, out_fmt: str = "f32",
                       out_seq_stride: int = 0):
    """One decode step: ca/za (and cb/zb) [B, c] rows of the token at position pos[b]
    ([B] int64; < 0 skips b).  The token that completes block i writes entry i to row
    b*out_seq_stride + i of `out` (e.g. a cache [B, N, row])."""
    B, c = ca.shape
    st = _lib().csa2_compress_step(ctx(ca.device.index), _p(ca), _p(za), _p(cb), _p(zb), _dt(ca), _p(ba), _p(bb),
                                   B, c, m, _p(pos), _p(state), rope_base, flags, _vp(out.data_ptr()),
                                   _out_dt(out, out_fmt), out_seq_stride, _stream(ca))
    _check("csa2_compress_step", st)
    return out


def csa2_compress_state_seed(ca, za, m: int, state, cb=None, zb=None):
    """Seed the state from the first n tokens of each sequence ([B, n, c] rows)."""
    B, n, c = ca.shape
    st = _lib().csa2_compress_state_seed(ctx(ca.device.index), _p(ca), _p(za), _p(cb), _p(zb), _dt(ca), B, n, c, m,
                                         _p(state), _stream(ca))
    _check("csa2_compress_state_seed", st)


def csa2_compress(ca, za, m: int, cb=None, zb=None, ba=None, bb=None, prev_cb=None, prev_zb=None,
                  pos0=0, rope_base: float = 10000.0, flags: int = 0, out_fmt: str = "f32",
                  out: Optional[torch.Tensor] = None, out_seq_stride: Optional[int] = None) -> torch.Tensor:
    """Compressed entries of one token stream [n, c] or a batch [B, n, c] -> [.., n/m, c]
    (out_fmt 'f32', 'bf16') or packed FP4 / MXFP4 rows ('fp4', 'mxfp4').  pos0: int or [B] int64 tensor
    (position of each stream's first token).  With `out` and `out_seq_stride`, entry i
    of stream b goes to row b*out_seq_stride + i of `out` (e.g. into a cache)."""
    batched = ca.dim() == 3
    B, n, c = (ca.shape if batched else (1, *ca.shape))
    n_ent = n // m
    if out is None:
        shape = (B, n_ent) if batched else (n_ent,)
        out = _alloc_rows(shape, c, out_fmt, ca.device)
    oss = n_ent if out_seq_stride is None else out_seq_stride
    out_dt = _out_dt(out, out_fmt)
    if isinstance(pos0, torch.Tensor):
        pos_t = pos0.to(device=ca.device, dtype=torch.int64).contiguous()
    else:
        pos_t = torch.full((B,), int(pos0), dtype=torch.int64, device=ca.device)
    st = _lib().csa2_compress(ctx(ca.device.index), _p(ca), _p(za), _p(cb), _p(zb), _dt(ca), _p(ba), _p(bb),
                              _p(prev_cb), _p(prev_zb), B, n, c, m, _p(pos_t), rope_base, flags,
                              _vp(out.data_ptr()), out_dt, oss, _stream(ca))
    _check("csa2_compress", st)
    return out


def csa2_visible_entries(q_pos: torch.Tensor, m: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Entries visible to each query position, floor(t / m) (0 for t < 0): the causal
    rule of the compressed cache (DSA-to-CSA/HCA page, «因果边界与短滑窗»).  q_pos:
    int64 device tensor of any shape; returns the same shape."""
    if q_pos.dtype != torch.int64 or not q_pos.is_cuda:
        raise ValueError("q_pos must be an int64 CUDA tensor")
    q_pos = q_pos.contiguous()
    if out is None:
        out = alloc(tuple(q_pos.shape), dtype=torch.int64, device=q_pos.device)
    if out.shape != q_pos.shape or out.dtype != torch.int64 or not out.is_contiguous():
        raise ValueError("out must be a contiguous int64 tensor shaped like q_pos")
    st = _lib().csa2_visible_entries(ctx(q_pos.device.index), _p(q_pos), q_pos.numel(), int(m), _p(out),
                                     _stream(q_pos))
    _check("csa2_visible_entries", st)
    return out


def csa2_index_score_mxq(qI, w, kI, n_visible, block: int = 8, scores: Optional[torch.Tensor] = None,
                         block_max: Optional[torch.Tensor] = None, want_scores: bool = True,
                         want_block_max: bool = False, block_hist: Optional[torch.Tensor] = None,
                         q_mx_out: Optional[torch.Tensor] = None):
    """Full scan on the FP4 QK path from a bf16 indexer query qI [B,Q,64,128], packed to
    MXFP4 inside the scan (by csa2_fp4_pack's rule; the packed bytes go to q_mx_out
    [B,Q,64,68] uint8 if given); kI [B,N,68] MXFP4.  Outputs as csa2_index_score's full
    scan.  Returns (scores, block_max)."""
    if qI.dtype != torch.bfloat16 or kI.dtype != torch.uint8:
        raise ValueError("csa2_index_score_mxq takes a bf16 query and MXFP4 keys")
    B, Q, H_I, d = qI.shape
    N = kI.shape[1]
    if want_scores and scores is None:
        scores = alloc((B, Q, N), dtype=torch.float32, device=qI.device)
    if want_block_max and block_max is None:
        block_max = alloc((B, Q, (N + block - 1) // block), dtype=torch.float32, device=qI.device)
    if q_mx_out is not None and (q_mx_out.dtype != torch.uint8 or q_mx_out.shape != (B, Q, H_I, mxfp4_row_bytes(d))):
        raise ValueError("q_mx_out must be uint8 [B, Q, H_I, 68]")
    st = _lib().csa2_index_score_mxq(ctx(qI.device.index), _p(qI), _p(w), _p(kI), B, Q, N, H_I, d, _p(n_visible),
                                     block, _p(scores) if want_scores else None, _p(block_max), _p(block_hist),
                                     _p(q_mx_out), _stream(qI))
    _check("csa2_index_score_mxq", st)
    return scores, block_max


def csa2_index_score(qI, w, kI, n_visible, k_fmt: Optional[int] = None, pool=None, block: int = 8,
                     scores: Optional[torch.Tensor] = None, block_max: Optional[torch.Tensor] = None,
                     want_scores: bool = True, want_block_max: bool = False,
                     block_hist: Optional[torch.Tensor] = None):
    """qI [B,Q,H_I,d] (f32/bf16) or [B,Q,H_I,68] uint8 (MXFP4, d = 128), w [B,Q,H_I],
    kI [B,N,d] (f32/bf16) or [B,N,row_bytes] uint8 (MXFP4), n_visible [B,Q] int64.
    MXFP4 queries over MXFP4 keys run the QK product in FP4 on the tensor cores.
    block_hist ([B,Q,BLOCK_HIST_BINS] int32 storage, full scan with block_max only)
    receives the block maxima's summary for csa2_block_pool.
    Returns (scores, block_max); either may be None."""
    B, Q, H_I, d = qI.shape
    if qI.dtype == torch.uint8:
        q_dt, d = MXFP4_E8M0x32, 128
    else:
        q_dt = _dt(qI)
    N = kI.shape[1]
    if kI.dtype == torch.uint8:
        k_dt = MXFP4_E8M0x32 if k_fmt is None else k_fmt
    else:
        k_dt = _dt(kI)
    n_pool = 0
    if pool is not None:
        n_pool = pool.shape[-1]
        if scores is None:
            scores = alloc((B, Q, n_pool * block), dtype=torch.float32, device=qI.device)
    else:
        if want_scores and scores is None:
            scores = alloc((B, Q, N), dtype=torch.float32, device=qI.device)
        if want_block_max and block_max is None:
            block_max = alloc((B, Q, (N + block - 1) // block), dtype=torch.float32, device=qI.device)
    st = _lib().csa2_index_score(ctx(qI.device.index), _p(qI), q_dt, _p(w), _p(kI), k_dt, B, Q, N, H_I, d,
                                 _p(n_visible), _p(pool), n_pool, block, _p(scores), _p(block_max),
                                 _p(block_hist), _stream(qI))
    _check("csa2_index_score", st)
    return scores, block_max


def csa2_topk_workspace_bytes(rows: int, n: int, k: int, device: Optional[int] = None) -> int:
    return int(_lib().csa2_topk_workspace_bytes(ctx(device), rows, n, k))


def csa2_block_pool_workspace_bytes(rows: int, ld: int, n_keep: int, device: Optional[int] = None) -> int:
    return int(_lib().csa2_block_pool_workspace_bytes(ctx(device), rows, ld, n_keep))


def _ws(nbytes: int, device) -> torch.Tensor:
    return alloc(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def csa2_topk(scores, n_visible, k: int, pool=None, block: int = 8, want_scores: bool = False,
              out_idx: Optional[torch.Tensor] = None, out_score: Optional[torch.Tensor] = None,
              ws: Optional[torch.Tensor] = None):
    """scores [..., n] -> (idx [..., k] int32 ascending, -1 padded; matching scores or None).
    `ws` is the split-row workspace (allocated here when not given)."""
    n = scores.shape[-1]
    rows = scores.numel() // n if n else 0
    lead = scores.shape[:-1]
    if out_idx is None:
        out_idx = alloc((*lead, k), dtype=torch.int32, device=scores.device)
    if want_scores and out_score is None:
        out_score = alloc((*lead, k), dtype=torch.float32, device=scores.device)
    n_pool = pool.shape[-1] if pool is not None else 0
    if ws is None:
        ws = _ws(csa2_topk_workspace_bytes(rows, n, k, scores.device.index) if rows else 0, scores.device)
    st = _lib().csa2_topk(ctx(scores.device.index), _p(scores), rows, n, n, _p(n_visible), _p(pool), n_pool, block,
                          k, _p(out_idx), _p(out_score), _p(ws), ws.numel(), _stream(scores))
    _check("csa2_topk", st)
    return out_idx, out_score


def csa2_block_pool(block_max, n_visible, block: int = 8, n_keep: int = 2048,
                    out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    block_hist: Optional[torch.Tensor] = None, n_top: int = 0,
                    out_top: Optional[torch.Tensor] = None):
    """The pool ([..., n_keep] int32).  With n_top > 0 also the n_top best blocks
    ([..., n_top] int32, ascending): returns (pool, top) then."""
    ld = block_max.shape[-1]
    rows = block_max.numel() // ld if ld else 0
    if out is None:
        out = alloc((*block_max.shape[:-1], n_keep), dtype=torch.int32, device=block_max.device)
    if n_top > 0 and out_top is None:
        out_top = alloc((*block_max.shape[:-1], n_top), dtype=torch.int32, device=block_max.device)
    if ws is None:
        ws = _ws(csa2_block_pool_workspace_bytes(rows, ld, n_keep, block_max.device.index) if rows else 0,
                 block_max.device)
    st = _lib().csa2_block_pool(ctx(block_max.device.index), _p(block_max), _p(block_hist), rows, ld, _p(n_visible),
                                block, n_keep, _p(out), _p(out_top) if n_top > 0 else None, n_top, _p(ws),
                                ws.numel(), _stream(block_max))
    _check("csa2_block_pool", st)
    return (out, out_top) if n_top > 0 else out


def csa2_block_hist(block_max, n_visible, block: int = 8, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The histogram of block maxima [..., ld] that csa2_block_pool / csa2_pool_topk take
    ([..., BLOCK_HIST_BINS] int32 storage)."""
    ld = block_max.shape[-1]
    rows = block_max.numel() // ld if ld else 0
    if out is None:
        out = alloc((*block_max.shape[:-1], BLOCK_HIST_BINS), dtype=torch.int32, device=block_max.device)
    st = _lib().csa2_block_hist(ctx(block_max.device.index), _p(block_max), rows, ld, _p(n_visible), block, _p(out),
                                _stream(block_max))
    _check("csa2_block_hist", st)
    return out


def csa2_pool_topk(block_max, block_hist, scores, n_visible, k: int, block: int = 8, n_keep: int = 2048,
                   out: Optional[torch.Tensor] = None, out_idx: Optional[torch.Tensor] = None,
                   out_score: Optional[torch.Tensor] = None, want_scores: bool = False):
    """Pool and top-k of a Full decode layer from the scan's block maxima [..., ld],
    their histogram [..., BLOCK_HIST_BINS] and the full scores [..., n_ent]:
    returns (pool [..., n_keep], idx [..., k], scores of idx or None)."""
    ld = block_max.shape[-1]
    rows = block_max.numel() // ld if ld else 0
    lead = block_max.shape[:-1]
    n_ent = scores.shape[-1]
    if out is None:
        out = alloc((*lead, n_keep), dtype=torch.int32, device=block_max.device)
    if out_idx is None:
        out_idx = alloc((*lead, k), dtype=torch.int32, device=block_max.device)
    if want_scores and out_score is None:
        out_score = alloc((*lead, k), dtype=torch.float32, device=block_max.device)
    st = _lib().csa2_pool_topk(ctx(block_max.device.index), _p(block_max), _p(block_hist), _p(scores), rows, ld, n_ent,
                               _p(n_visible), block, n_keep, k, _p(out), _p(out_idx), _p(out_score),
                               _stream(block_max))
    _check("csa2_pool_topk", st)
    return out, out_idx, out_score


def csa2_sparse_attn_workspace_bytes(B: int, Q: int, H: int, k: int, window: int,
                                     device: Optional[int] = None, N: int = 0, swa_cap: int = 0) -> int:
    return int(_lib().csa2_sparse_attn_workspace_bytes(ctx(device), B, Q, H, k, window, N, swa_cap))


def csa2_sparse_attn(q, kv, idx, swa, q_pos, sink=None, window: int = 128, swa_pos0: int = 0,
                     kv_fmt: Optional[int] = None, rope_base: float = 10000.0, flags: int = ATTN_DEFAULT,
                     out_dtype=None, want_lse: bool = False, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None):
    """q [B,Q,H,c]; kv [B,N,c] (f32/bf16) or [B,N,row_bytes] uint8 (FP4); idx [B,Q,k] int32;
    swa [B,cap,c]; q_pos [B,Q] int64.  Returns (out [B,Q,H,c], lse [B,Q,H] or None).
    `ws` is the split-key workspace (allocated here when not given)."""
    B, Q, H, c = q.shape
    k = idx.shape[-1] if idx is not None else 0
    N = kv.shape[1] if kv is not None else 0
    kv_dt = (FP4_E4M3x16 if kv_fmt is None else kv_fmt) if kv is not None and kv.dtype == torch.uint8 else \
        (_dt(kv) if kv is not None else F32)
    swa_cap = swa.shape[1] if swa is not None else 0
    swa_dt = _dt(swa) if swa is not None else F32
    if out is None:
        out = alloc((B, Q, H, c), dtype=out_dtype or q.dtype, device=q.device)
    if want_lse and lse is None:
        lse = alloc((B, Q, H), dtype=torch.float32, device=q.device)
    if ws is None:
        nb = csa2_sparse_attn_workspace_bytes(B, Q, H, k, window, q.device.index, N=N, swa_cap=swa_cap)
        ws = alloc(max(nb, 16), dtype=torch.uint8, device=q.device)
    st = _lib().csa2_sparse_attn(ctx(q.device.index), _p(q), _dt(q), _p(kv), kv_dt, N, _p(idx), k, _p(swa), swa_dt,
                                 swa_cap, swa_pos0, window, _p(q_pos), _p(sink), B, Q, H, c, rope_base, flags,
                                 _p(out), _dt(out), _p(lse), _p(ws), ws.numel() * ws.element_size(), _stream(q))
    _check("csa2_sparse_attn", st)
    return out, lse


def csa2_attn_prepare(q, q_pos, ws: torch.Tensor, k: int, window: int = 128, N: int = 0, swa_cap: int = 0,
                      rope_base: float = 10000.0, flags: int = ATTN_DEFAULT) -> None:
    """The query half of a later csa2_sparse_attn / csa2_dense_attn call with the same
    sizes, flags | ATTN_PREPARED and the same workspace `ws` (q [B,Q,H<=64,c])."""
    B, Q, H, c = q.shape
    st = _lib().csa2_attn_prepare(ctx(q.device.index), _p(q), _dt(q), _p(q_pos), B, Q, H, c, k, window, N, swa_cap,
                                  rope_base, flags, _p(ws), ws.numel() * ws.element_size(), _stream(q))
    _check("csa2_attn_prepare", st)


def csa2_dense_attn(q, kv, n_visible, k_max: int, swa, q_pos, sink=None, window: int = 128, swa_pos0: int = 0,
                    kv_fmt: Optional[int] = None, rope_base: float = 10000.0, flags: int = ATTN_DEFAULT,
                    out_dtype=None, want_lse: bool = False, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None):
    """HCA attention: each query over compressed entries 0 .. n_visible[b,q]-1 (all it
    can see) plus the window.  n_visible [B,Q] int64 <= k_max; otherwise as
    csa2_sparse_attn."""
    B, Q, H, c = q.shape
    N = kv.shape[1] if kv is not None else 0
    kv_dt = (FP4_E4M3x16 if kv_fmt is None else kv_fmt) if kv is not None and kv.dtype == torch.uint8 else \
        (_dt(kv) if kv is not None else F32)
    swa_cap = swa.shape[1] if swa is not None else 0
    swa_dt = _dt(swa) if swa is not None else F32
    if out is None:
        out = alloc((B, Q, H, c), dtype=out_dtype or q.dtype, device=q.device)
    if want_lse and lse is None:
        lse = alloc((B, Q, H), dtype=torch.float32, device=q.device)
    if ws is None:
        nb = csa2_sparse_attn_workspace_bytes(B, Q, H, k_max, window, q.device.index, N=N, swa_cap=swa_cap)
        ws = alloc(max(nb, 16), dtype=torch.uint8, device=q.device)
    st = _lib().csa2_dense_attn(ctx(q.device.index), _p(q), _dt(q), _p(kv), kv_dt, N, _p(n_visible), k_max, _p(swa),
                                swa_dt, swa_cap, swa_pos0, window, _p(q_pos), _p(sink), B, Q, H, c, rope_base, flags,
                                _p(out), _dt(out), _p(lse), _p(ws), ws.numel() * ws.element_size(), _stream(q))
    _check("csa2_dense_attn", st)
    return out, lse


def csa2_sparse_attn_noalloc(q, kv, idx, swa, q_pos, out: torch.Tensor, sink=None, window: int = 128,
                             swa_pos0: int = 0, kv_fmt: Optional[int] = None, rope_base: float = 10000.0,
                             flags: int = ATTN_DEFAULT, lse: Optional[torch.Tensor] = None):
    """csa2_sparse_attn without a workspace, for callers that may not allocate device
    memory: the library keeps the partial results in its own fixed device array.
    The caller passes every tensor, outputs included; nothing is allocated here."""
    B, Q, H, c = q.shape
    # the kernels write B*Q*H rows of c values (and B*Q*H lse values): a smaller
    # buffer would be overrun, so its shape, dtype and device are checked first
    if tuple(out.shape) != (B, Q, H, c) or out.device != q.device or out.dtype not in (torch.float32,
                                                                                      torch.bfloat16):
        raise ValueError(f"out must be a float32/bfloat16 tensor of shape {(B, Q, H, c)} on {q.device}")
    if lse is not None and (tuple(lse.shape) != (B, Q, H) or lse.dtype != torch.float32 or lse.device != q.device):
        raise ValueError(f"lse must be None or a float32 tensor of shape {(B, Q, H)} on {q.device}")
    k = idx.shape[-1] if idx is not None else 0
    N = kv.shape[1] if kv is not None else 0
    kv_dt = (FP4_E4M3x16 if kv_fmt is None else kv_fmt) if kv is not None and kv.dtype == torch.uint8 else \
        (_dt(kv) if kv is not None else F32)
    swa_cap = swa.shape[1] if swa is not None else 0
    swa_dt = _dt(swa) if swa is not None else F32
    st = _lib().csa2_sparse_attn_noalloc(ctx(q.device.index), _p(q), _dt(q), _p(kv), kv_dt, N, _p(idx), k, _p(swa),
                                         swa_dt, swa_cap, swa_pos0, window, _p(q_pos), _p(sink), B, Q, H, c,
                                         rope_base, flags, _p(out), _dt(out), _p(lse), _stream(q))
    _check("csa2_sparse_attn_noalloc", st)
    return out, lse
