"""gc_select_if_noalloc, the entry point that allocates nothing.

Some callers cannot allocate device memory where they need a compaction (a
plugin inside a framework that owns the device memory budget, a loop that
must not pay for cudaMalloc's possible device synchronisation), so this
variant of select-if keeps its scratch in a fixed array inside the library.
Its results must be those of gc_select_if, call after call: the shared
array keeps the previous call's contents, and each call must clear what has
to start at zero.  This file sorts last so that a run stopping at the first
failure has run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from partition_pass_tile_gb300 import gc, synth

pytestmark = pytest.mark.gpu


def _host(t):
    return t.view(torch.int32).cpu().numpy().view(np.uint32) if t.dtype == torch.uint32 \
        else t.cpu().numpy()


def _entry():
    f = gc.load().gc_select_if_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def test_noalloc_matches_select_if_on_consecutive_calls():
    f = _entry()
    T = gc.tile_elements(gc.OP_SELECT_IF)
    # two calls in a row with different sizes, dtypes and predicates; the
    # second is smaller, so stale status words of the first lie beyond it
    cases = [(1_047_965, "remove_zeros", gc.NONZERO), (3 * T + 611, "uniform", gc.ODD)]
    stream = torch.cuda.current_stream()
    for n, kind, pred in cases:
        host = synth.remove_zeros(n, 1) if kind == "remove_zeros" else synth.uniform_i32(n, 3)
        x = torch.from_numpy(host).cuda()
        want_out, want_cnt = gc.select_if(x, pred)          # the existing entry point
        out = torch.full_like(x, -1)
        cnt = torch.full((1,), 7, dtype=torch.int32, device="cuda").view(torch.uint32)
        st = f(x.data_ptr(), out.data_ptr(), cnt.data_ptr(), n, gc.I32, pred, stream.cuda_stream)
        assert st == 0, gc.STATUS.get(st, st)
        torch.cuda.synchronize()
        m = int(_host(cnt)[0])
        assert m == int(_host(want_cnt)[0])
        assert np.array_equal(_host(out)[:m], _host(want_out)[:m])   # integer work: bit-exact


def test_noalloc_rejects_sizes_beyond_its_array():
    f = _entry()
    # validation happens on the host before any device work: fake pointers suffice
    st = f(0x10000000, 0x20000000, 0x30000000, gc.NOALLOC_MAX_ELEMENTS + 1, gc.I32, gc.NONZERO,
           None)
    assert gc.STATUS[st] == "GC_ERR_INVALID_VALUE"
