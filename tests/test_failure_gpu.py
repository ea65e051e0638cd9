"""Failure detection on the GPU without faulting it.

A wait that can never be satisfied, planted through a gc_testing.h hook (a
look-back on tile 0, which no CTA takes; a start barrier whose counter is
marked as one that ran out) must give up after its time limit, record
GC_ERR_TIMEOUT in the workspace and let the kernel finish; the host reads the
status, and the same workspace and context then work normally.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import dev, host
from partition_pass_tile_gb300 import gc, synth

pytestmark = pytest.mark.gpu


def test_lookback_timeout_is_reported_and_recoverable(orc):
    T = gc.tile_elements(gc.OP_SELECT_IF)
    n = 6 * T + 11
    x = synth.uniform_i32(n, 21)
    xd = dev(x)
    ws = gc.workspace(gc.OP_SELECT_IF, n)
    out = torch.empty_like(xd)
    cnt = torch.empty(1, dtype=torch.uint32, device="cuda")
    st = gc.testing_select_if_skip_tile0(xd, "odd", out, cnt, ws, timeout_ns=20_000_000)
    assert st == 0
    torch.cuda.synchronize()            # the kernel finished: nothing hung
    assert gc.query_device_status(ws) == 6   # GC_ERR_TIMEOUT
    assert gc.query_device_status(ws) == 0   # read-and-clear
    # same workspace, same context: a normal call is right again
    out, cnt = gc.select_if(xd, "odd", ws=ws)
    want = orc.select_if(x, O.ODD)
    m = int(host(cnt)[0])
    assert m == want.shape[0] and np.array_equal(host(out)[:m], want)
    assert gc.query_device_status(ws) == 0


def test_testing_hook_rejects_single_tile():
    T = gc.tile_elements(gc.OP_SELECT_IF)
    x = torch.ones(T, dtype=torch.int32, device="cuda")
    ws = gc.workspace(gc.OP_SELECT_IF, T)
    st = gc.testing_select_if_skip_tile0(x, "odd", torch.empty_like(x),
                                         torch.empty(1, dtype=torch.uint32, device="cuda"), ws,
                                         timeout_ns=1_000_000)
    assert st == 1  # GC_ERR_INVALID_VALUE


def test_start_barrier_timeout_is_reported_and_recoverable(orc):
    n = 3_000_017  # several CTAs per SM's worth of tiles: the whole persistent grid
    x = synth.uniform_i32(n, 22)
    xd = dev(x)
    ws = gc.workspace(gc.OP_EXCLUSIVE_SCAN, n)
    out = torch.empty_like(xd)
    tot = torch.empty(1, dtype=torch.int32, device="cuda")
    st = gc.testing_exclusive_scan_stalled_barrier(xd, out, tot, ws, timeout_ns=5_000_000)
    assert st == 0
    torch.cuda.synchronize()
    assert gc.query_device_status(ws) == 6   # GC_ERR_TIMEOUT
    assert gc.query_device_status(ws) == 0   # read-and-clear, barrier words included
    want, _ = orc.exclusive_scan(x)
    for _ in range(2):  # the barrier completes again, call after call
        out, tot = gc.exclusive_scan(xd, ws=ws)
        assert np.array_equal(host(out), want)
        assert gc.query_device_status(ws) == 0
