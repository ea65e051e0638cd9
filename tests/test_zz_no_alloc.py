"""gc_select_if_noalloc, the entry point that allocates nothing.

Some callers cannot allocate device memory where they need a compaction: a
plugin inside a framework that owns the whole device memory budget, or a
loop that must not pay for cudaMalloc / cudaFree, which may synchronise the
device.  This variant of select-if therefore keeps its scratch in a fixed
array inside the library.  Its results must be the oracle's and those of
gc_select_if, call after call: the shared array keeps the previous call's
contents, and each call must clear what has to start at zero, on the
persistent path (status words cleared in the kernel) and on the
one-tile-per-CTA path (taken when the device refuses a cooperative grid,
forced here by a test hook; it clears the array with a memset) alike.
This file sorts last so that a run stopping at the first failure has run
every other test before it; it passes alone in a fresh process too.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import dev, host
from partition_pass_tile_gb300 import gc, synth

pytestmark = pytest.mark.gpu


def _entry():
    f = gc.load().gc_select_if_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _case(kind, n):
    if kind == "remove_zeros":
        return synth.remove_zeros(n, 1), gc.NONZERO
    if kind == "u32_odd":
        return synth.uniform_u32(n, 3), gc.ODD
    x = synth.scan_unit_f32(n, 2)
    x[synth.uniform_u32(n, 4) % 4 == 0] = 0.0
    x[synth.uniform_u32(n, 5) % 16 == 0] = -0.0
    return x, gc.NONZERO


def _call(f, x_host, pred, offset):
    """One call through the C ABI on an input `offset` elements into its
    allocation (offset 1: not 16-byte aligned), into an output prefilled
    with -1 bits; returns (count, output bits)."""
    xd = dev(x_host, offset)
    n = x_host.shape[0]
    big = torch.full((n + 4,), -1, dtype=torch.int32, device="cuda")
    out = big[:n]
    cnt = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    st = f(xd.data_ptr(), out.data_ptr(), cnt.data_ptr(), n, gc.dtype_code(xd), pred,
           stream.cuda_stream)
    assert st == 0, gc.STATUS.get(st, st)
    torch.cuda.synchronize()
    return int(cnt.item()), out.cpu().numpy().view(np.uint32), xd


def test_noalloc_matches_oracle_and_select_if_on_consecutive_calls(orc):
    f = _entry()
    T = gc.tile_elements(gc.OP_SELECT_IF)
    # Calls in a row with different sizes, dtypes, predicates and pointer
    # alignments: persistent, then one-tile-per-CTA (forced: the array's
    # memset path), then persistent again over the fallback's leftovers, and
    # smaller calls whose stale status words lie beyond them.
    cases = [("remove_zeros", 1_047_965, 0, False), ("u32_odd", 3 * T + 611, 1, True),
             ("f32_nonzero", 100_003, 0, False), ("remove_zeros", 2 * T + 5, 1, True),
             ("u32_odd", 5 * T, 2, False), ("f32_nonzero", 1_000, 1, True),
             ("remove_zeros", 1_047_965, 3, False)]
    for kind, n, offset, fallback in cases:
        x, pred = _case(kind, n)
        gc.testing_force_fallback(fallback)
        try:
            m, got, xd = _call(f, x, pred, offset)
        finally:
            gc.testing_force_fallback(False)
        want = orc.select_if(x, pred)                        # the oracle
        assert m == want.shape[0], (kind, n, offset)
        assert np.array_equal(got[:m], want.view(np.uint32)), (kind, n, offset)
        assert np.all(got[m:] == 0xFFFFFFFF)                 # nothing past the survivors
        ref_out, ref_cnt = gc.select_if(xd, pred)            # the entry point with a workspace
        assert int(host(ref_cnt)[0]) == m
        assert np.array_equal(host(ref_out)[:m].view(np.uint32), got[:m])
    assert gc.select_if_noalloc_status() == 0


def test_noalloc_empty_input_writes_zero():
    f = _entry()
    cnt = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    st = f(None, None, cnt.data_ptr(), 0, gc.I32, gc.NONZERO, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0


def test_noalloc_status_reports_a_stalled_barrier_and_recovers(orc):
    """A start barrier that never completes (planted on the host through the
    test hook): every wait gives up after 2 ms, the status query reports
    GC_ERR_TIMEOUT once and clears the barrier, and the next calls are exact."""
    n = 4 * gc.tile_elements(gc.OP_SELECT_IF) + 17
    x = synth.remove_zeros(n, 8)
    xd = dev(x)
    out = torch.empty_like(xd)
    cnt = torch.empty(1, dtype=torch.uint32, device="cuda")
    assert gc.testing_select_if_noalloc_stalled_barrier(xd, "nonzero", out, cnt, 2_000_000) == 0
    assert gc.select_if_noalloc_status() == 6     # GC_ERR_TIMEOUT
    assert gc.select_if_noalloc_status() == 0     # read once, then cleared
    want = orc.select_if(x, O.NONZERO)
    for _ in range(2):
        o2, c2 = gc.select_if_noalloc(xd, "nonzero")
        torch.cuda.synchronize()
        m = int(host(c2)[0])
        assert m == want.shape[0] and np.array_equal(host(o2)[:m], want)
        assert gc.select_if_noalloc_status() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    f = _entry()
    # validation happens on the host before any device work: fake pointers suffice
    st = f(0x10000000, 0x20000000, 0x30000000, gc.NOALLOC_MAX_ELEMENTS + 1, gc.I32, gc.NONZERO,
           None)
    assert gc.STATUS[st] == "GC_ERR_INVALID_VALUE"
