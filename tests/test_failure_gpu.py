"""Failure detection on the GPU without faulting it.

A look-back wait that can never be satisfied (tile 0 is never taken, planted
through the gc_testing.h hook) must give up after its time limit, record
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
