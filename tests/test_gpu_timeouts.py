"""Failure detection of the device waits: each wait of the library gives up
after one second, sets its dev_status flag and returns.  A self-test entry
point runs a wait that nothing will end (a radix-sort look-back on a tile no
CTA publishes; an mbarrier phase no copy completes); the flag must be set
and the context must stay usable (a normal step afterwards matches the
oracle).  Nothing faults, traps or hangs: the wait itself is bounded."""
import time

import numpy as np
import pytest
import torch

import workloads
from parity import check_full, run_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,flag", [(0, 0x4), (1, 0x20)])
def test_bounded_wait_gives_up_and_flags(kind, flag):
    from recsys_table_embedding_gb300.tbe import tbe_selftest_wait_limit
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    tbe_selftest_wait_limit(kind, st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st[1].item()) == flag
    assert 0.9 < dt < 30.0
    # the context still works
    wl = workloads.tiny()
    W0, G, m0 = wl.weights(), wl.grad_out(), wl.momentum()
    res = run_cuda(wl, W0, G, m0)
    check_full(wl, W0, G, m0, res)
    assert res["status"][1] == 0
