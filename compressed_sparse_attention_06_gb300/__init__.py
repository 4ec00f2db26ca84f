"""CSA2 compressed sparse attention hot path for GB300 (sm_103a).

`csa2` is the binding of the C ABI in libcsa2.so (include/csa2.h); `pipeline`
strings the entry points into the per-layer steps; `workloads` draws the seeded
synthetic inputs.  The library is loaded on first use and there is no other
implementation of the path: a missing libcsa2.so raises ImportError.
"""
from . import csa2, pipeline, workloads  # noqa: F401

__all__ = ["csa2", "pipeline", "workloads"]
