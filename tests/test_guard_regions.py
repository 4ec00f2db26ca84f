"""The guard-region checker used around every buffer of the GPU tests, exercised on
host memory: writes inside a buffer pass, a write one byte before or after it is
reported, and freed buffers are no longer checked."""
import pytest
import torch

from tests.helpers import GUARD_BYTES, GuardedAlloc


def test_inside_writes_pass_and_stray_writes_are_caught():
    ga = GuardedAlloc()
    a = ga.alloc((3, 5), torch.float32, "cpu")
    b = ga.alloc(7, torch.int64, "cpu")
    assert a.data_ptr() - a._guard_raw.data_ptr() == b.data_ptr() - b._guard_raw.data_ptr() == GUARD_BYTES
    a.fill_(1.5)
    b.fill_(-1)
    ga.verify("inside")
    assert ga.checked == 2
    a._guard_raw[GUARD_BYTES - 1] = 0                     # one byte before the buffer
    with pytest.raises(AssertionError, match="outside"):
        ga.verify("before")
    a._guard_raw[GUARD_BYTES - 1] = 0xA5
    b._guard_raw[GUARD_BYTES + 7 * 8] = 0                 # one byte after the buffer
    with pytest.raises(AssertionError, match="outside"):
        ga.verify("after")


def test_freed_buffers_are_dropped():
    ga = GuardedAlloc()
    a = ga.alloc((4,), torch.uint8, "cpu")
    a._guard_raw[0] = 0
    del a
    ga.verify("freed")
    assert ga.live == []
