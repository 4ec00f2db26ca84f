import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def golden():
    return load_golden


@pytest.fixture(autouse=True)
def _guarded_buffers(request, monkeypatch):
    """GPU tests: every buffer the binding allocates gets guard bytes before and after
    it, checked on the host after every library call and at the end of the test."""
    if request.node.get_closest_marker("gpu") is None:
        yield None
        return
    import torch
    if not torch.cuda.is_available():
        yield None
        return
    from compressed_sparse_attention_06_gb300 import csa2 as C
    from tests.helpers import GuardedAlloc
    ga = GuardedAlloc()
    check = C._check

    def checked(fn, st):
        check(fn, st)
        if ga.live and not fn.endswith("_workspace_bytes"):
            ga.verify(fn)

    monkeypatch.setattr(C, "alloc", ga.alloc)
    monkeypatch.setattr(C, "_check", checked)
    yield ga
    ga.verify("end of test")
