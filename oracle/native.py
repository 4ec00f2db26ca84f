"""The C++ restatement of the oracle (csa2_oracle.cpp) and its build.

TEST INFRASTRUCTURE, like csa2_oracle.py: only the tests, the smoke check and the
bench's CPU-baseline / reference leg load this.  build() compiles
libcsa2_oracle.so beside the source with the host compiler (g++ -O2 -std=c++17,
no architecture flags, so the same source builds on x86-64 and Arm hosts).

The wrappers take and return numpy arrays in float64 / int64 and mirror the
numpy oracle's functions of the same names; the tests hold the two to each other.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csa2_oracle.cpp")
LIB = os.path.join(HERE, "libcsa2_oracle.so")

QNORM, KVNORM, ROPE = 1, 2, 4
ROPE_BASE = 10000.0

_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = os.environ.get("CXX", "g++")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", "-o", tmp, SRC]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


_D = ctypes.POINTER(ctypes.c_double)
_F = ctypes.POINTER(ctypes.c_float)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I64 = ctypes.POINTER(ctypes.c_int64)
_i, _i64, _d = ctypes.c_int, ctypes.c_int64, ctypes.c_double

_SIGS = {
    "csa2o_version": ([], _i),
    "csa2o_e2m1_value": ([_i], _d),
    "csa2o_e4m3_value": ([_i], _d),
    "csa2o_e8m0_value": ([_i], _d),
    "csa2o_e2m1_encode": ([_d], _i),
    "csa2o_e4m3_encode": ([_d], _i),
    "csa2o_nvfp4_pack": ([_F, _i64, _i, _U8], None),
    "csa2o_nvfp4_unpack": ([_U8, _i64, _i, _D], None),
    "csa2o_mxfp4_pack": ([_F, _i64, _i, _U8], None),
    "csa2o_mxfp4_unpack": ([_U8, _i64, _i, _D], None),
    "csa2o_compress": ([_D, _D, _i64, _i, _i, _D, _D, _D, _D, _D, _D, _D], None),
    "csa2o_compress_write": ([_D, _i64, _i, _i, _i, _i64, _d], None),
    "csa2o_rms_norm": ([_D, _i64, _i], None),
    "csa2o_rope": ([_D, _i64, _i, _i64, _i, _d], None),
    "csa2o_index_score": ([_D, _D, _D, _i64, _i64, _i, _i, _D], None),
    "csa2o_topk": ([_D, _i64, _i, _I64], None),
    "csa2o_block_max": ([_D, _i64, _i, _D], None),
    "csa2o_block_pool": ([_D, _i64, _i, _i, _I64], None),
    "csa2o_reindex_topk": ([_D, _I64, _i, _i64, _i, _i, _I64], None),
    "csa2o_attend": ([_D, _D, _i64, _i, _i, _i64, _D, _i, _d, _D, _D], None),
    "csa2o_sparse_attn": ([_D, _D, _I64, _i, _D, _i64, _i64, _i64, _D, _i, _i, _i, _i, _d, _D, _D], None),
    "csa2o_decode_query_fp4": ([_U8, _i64, _i64, _U8, _D, _i, _i, _i, _i, _I64, _U8, _i64, _D, _i, _D, _i64,
                                _i64, _i64, _D, _i, _d, _i, _D, _D, _I64], _i),
}


def lib():
    """The loaded library (built first if needed)."""
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray], ptr):
    return None if a is None else a.ctypes.data_as(ptr)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def e2m1_value(code: int) -> float:
    return lib().csa2o_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().csa2o_e4m3_value(int(code))


def e8m0_value(code: int) -> float:
    return lib().csa2o_e8m0_value(int(code))


def e2m1_encode(x: float) -> int:
    return lib().csa2o_e2m1_encode(float(x))


def e4m3_encode(x: float) -> int:
    return lib().csa2o_e4m3_encode(float(x))


def nvfp4_pack(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, c = x.shape
    out = np.empty((rows, c // 2 + c // 16), dtype=np.uint8)
    lib().csa2o_nvfp4_pack(_p(x, _F), rows, c, _p(out, _U8))
    return out


def nvfp4_unpack(b, c: int = 512) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty((b.shape[0], c))
    lib().csa2o_nvfp4_unpack(_p(b, _U8), b.shape[0], c, _p(out, _D))
    return out


def mxfp4_pack(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, d = x.shape
    out = np.empty((rows, d // 2 + d // 32), dtype=np.uint8)
    lib().csa2o_mxfp4_pack(_p(x, _F), rows, d, _p(out, _U8))
    return out


def mxfp4_unpack(b, d: int = 128) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty((b.shape[0], d))
    lib().csa2o_mxfp4_unpack(_p(b, _U8), b.shape[0], d, _p(out, _D))
    return out


def compress(Ca, Za, m: int, Ba=None, Cb=None, Zb=None, Bb=None, prev_Cb=None, prev_Zb=None) -> np.ndarray:
    Ca, Za, Ba, Cb, Zb, Bb, prev_Cb, prev_Zb = map(_f64, (Ca, Za, Ba, Cb, Zb, Bb, prev_Cb, prev_Zb))
    n, c = Ca.shape
    if n % m:
        raise ValueError("n must be a multiple of m")
    out = np.empty((n // m, c))
    lib().csa2o_compress(_p(Ca, _D), _p(Za, _D), n, c, m, _p(Ba, _D), _p(Cb, _D), _p(Zb, _D), _p(Bb, _D),
                         _p(prev_Cb, _D), _p(prev_Zb, _D), _p(out, _D))
    return out


def compress_write(E, flags: int, m: int, pos0: int = 0, base: float = ROPE_BASE) -> np.ndarray:
    """The f64 part of the write epilogue (RMSNorm, RoPE); packing is nvfp4_pack."""
    E = np.array(E, dtype=np.float64, copy=True, order="C")
    lib().csa2o_compress_write(_p(E, _D), E.shape[0], E.shape[1], flags & 3, m, pos0, base)
    return E


def rms_norm(x) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    c = x.shape[-1]
    lib().csa2o_rms_norm(_p(x, _D), x.size // c, c)
    return x


def rope(x, pos: int, inverse: bool = False, base: float = ROPE_BASE) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True, order="C")
    c = x.shape[-1]
    lib().csa2o_rope(_p(x, _D), x.size // c, c, int(pos), int(inverse), base)
    return x


def index_score(qI, w, KI, n_visible: int) -> np.ndarray:
    qI, w, KI = _f64(qI), _f64(w), _f64(KI)
    H, d = qI.shape
    out = np.empty(KI.shape[0])
    lib().csa2o_index_score(_p(qI, _D), _p(w, _D), _p(KI, _D), KI.shape[0], int(n_visible), H, d, _p(out, _D))
    return out


def topk(scores, n_visible: int, k: int) -> np.ndarray:
    s = _f64(scores)
    out = np.empty(k, dtype=np.int64)
    lib().csa2o_topk(_p(s, _D), int(n_visible), k, _p(out, _I64))
    return out


def block_max(scores, n_visible: int, block: int = 8) -> np.ndarray:
    s = _f64(scores)
    V = int(n_visible)
    out = np.empty((V + block - 1) // block if V > 0 else 0)
    lib().csa2o_block_max(_p(s, _D), V, block, _p(out, _D))
    return out


def block_pool(bmax, n_visible: int, block: int = 8, n_keep: int = 2048) -> np.ndarray:
    bm = _f64(bmax)
    out = np.empty(n_keep, dtype=np.int64)
    lib().csa2o_block_pool(_p(bm, _D), int(n_visible), block, n_keep, _p(out, _I64))
    return out


def reindex_topk(full_scores, pool_blocks, n_visible: int, k: int, block: int = 8) -> np.ndarray:
    s = _f64(full_scores)
    pool = np.ascontiguousarray(pool_blocks, dtype=np.int64)
    out = np.empty(k, dtype=np.int64)
    lib().csa2o_reindex_topk(_p(s, _D), _p(pool, _I64), pool.shape[0], int(n_visible), k, block, _p(out, _I64))
    return out


def attend(q, keys, t: int, sink=None, flags: int = QNORM | KVNORM | ROPE, base: float = ROPE_BASE):
    """(o [H, c], lse [H]) of one query over the given rows."""
    q, keys, sink = _f64(q), _f64(keys), _f64(sink)
    H, c = q.shape
    keys = keys.reshape(-1, c)
    out = np.empty((H, c))
    lse = np.empty(H)
    lib().csa2o_attend(_p(q, _D), _p(keys, _D), keys.shape[0], H, c, int(t), _p(sink, _D), flags, base,
                       _p(out, _D), _p(lse, _D))
    return out, lse


def sparse_attn(q, kv_entries, idx, swa, swa_pos0: int, t: int, sink=None, window: int = 128,
                flags: int = QNORM | KVNORM | ROPE, base: float = ROPE_BASE):
    q, kv, swa, sink = _f64(q), _f64(kv_entries), _f64(swa), _f64(sink)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    H, c = q.shape
    out = np.empty((H, c))
    lse = np.empty(H)
    lib().csa2o_sparse_attn(_p(q, _D), _p(kv, _D), _p(idx, _I64), idx.shape[0], _p(swa, _D), swa.shape[0],
                            swa_pos0, int(t), _p(sink, _D), window, H, c, flags, base, _p(out, _D), _p(lse, _D))
    return out, lse


def decode_query_fp4(ki, V: int, qI_mx, w, kv_ids, kv_rows, q, swa, swa_pos0: int, t: int, sink=None, *,
                     block: int = 8, n_keep: int = 2048, k: int = 512, window: int = 128,
                     base: float = ROPE_BASE, threads: Optional[int] = None):
    """One Full-mode decode query over FP4 caches (MXFP4 indexer rows ki [N, 68], the
    packed indexer query qI_mx [H_I, 68], the FP4 main-KV rows kv_rows [n, 288] of the
    ascending ids kv_ids, which must hold every selected id).  Returns (o, lse, idx)."""
    ki = np.ascontiguousarray(ki, dtype=np.uint8)
    qI_mx = np.ascontiguousarray(qI_mx, dtype=np.uint8)
    w, q, swa, sink = _f64(w), _f64(q), _f64(swa), _f64(sink)
    kv_ids = np.ascontiguousarray(kv_ids, dtype=np.int64)
    kv_rows = np.ascontiguousarray(kv_rows, dtype=np.uint8)
    H, c = q.shape
    out = np.empty((H, c))
    lse = np.empty(H)
    idx = np.empty(k, dtype=np.int64)
    nt = threads or os.cpu_count() or 1
    rc = lib().csa2o_decode_query_fp4(_p(ki, _U8), ki.shape[0], int(V), _p(qI_mx, _U8), _p(w, _D), qI_mx.shape[0],
                                      block, n_keep, k, _p(kv_ids, _I64), _p(kv_rows, _U8), kv_ids.shape[0],
                                      _p(q, _D), H, _p(swa, _D), swa.shape[0], swa_pos0, int(t), _p(sink, _D),
                                      window, base, nt, _p(out, _D), _p(lse, _D), _p(idx, _I64))
    if rc != 0:
        raise ValueError("a selected main-KV row was not provided")
    return out, lse, idx
