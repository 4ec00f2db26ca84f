"""The C-ABI library builds for sm_103a, loads, and exports every symbol declared in
include/csa2.h.  Host-only: no kernel is launched here."""
import ctypes
import os
import re

import pytest
import torch

from compressed_sparse_attention_06_gb300 import build_lib
from compressed_sparse_attention_06_gb300 import csa2 as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return C.load()


def test_header_declares_the_path():
    names = _declared()
    for n in ("csa2_compress", "csa2_index_score", "csa2_topk", "csa2_block_pool", "csa2_sparse_attn",
              "csa2_fp4_pack", "csa2_fp4_unpack"):
        assert n in names
    assert sorted(C.EXPORTS) == names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for s in range(6):
        assert lib.csa2_status_string(s)
    assert lib.csa2_status_string(99) == b"unknown status"
    assert lib.csa2_version() >= 1


def test_host_validation_rejects_before_launch(lib):
    # a NULL context is rejected on the host; nothing touches a device
    assert lib.csa2_topk(None, None, 1, 8, 8, None, None, 0, 8, 4, None, None, None, 0, None) == C.ERR_INVALID_ARG
    assert lib.csa2_block_pool(None, None, None, 1, 8, None, 8, 16, None, None, 0, None, 0, None) == \
        C.ERR_INVALID_ARG
    assert lib.csa2_index_score(None, None, 0, None, None, 0, 1, 1, 8, 64, 128, None, None, 0, 8, None, None, None,
                                None) == C.ERR_INVALID_ARG
    assert lib.csa2_topk_workspace_bytes(None, 8, 16384, 512) == 0
    assert lib.csa2_sparse_attn(None, None, 0, None, 0, 0, None, 0, None, 0, 0, 0, 0, None, None, 1, 1, 64, 512,
                                10000.0, 7, None, 0, None, None, 0, None) == C.ERR_INVALID_ARG
    assert lib.csa2_sparse_attn_workspace_bytes(None, 8, 1, 64, 512, 128, 1000, 128) == 0
    assert lib.csa2_visible_entries(None, None, 4, 2, None, None) == C.ERR_INVALID_ARG
    assert lib.csa2_ctx_destroy(None) == C.ERR_INVALID_ARG
    assert lib.csa2_ctx_check(None, None) == C.ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_ctx_create_without_gpu_reports_cuda_error(lib):
    h = ctypes.c_void_p()
    assert lib.csa2_ctx_create(0, ctypes.byref(h)) in (C.ERR_CUDA, C.ERR_INVALID_ARG)
    assert not h.value


def test_library_is_sm103a_only():
    # the build passes exactly one -gencode, for sm_103a
    assert build_lib.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
