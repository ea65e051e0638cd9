"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, sizes workspaces, and rejects bad arguments on the host
before any CUDA call (every call below fails validation, so nothing reaches
the device)."""

import ctypes
import os
import re
import subprocess

import pytest

from partition_pass_tile_gb300 import build as gc_build
from partition_pass_tile_gb300 import gc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gc_build.build()
    return gc.load()


def declared_functions():
    names = set()
    for h in ("gc.h", "gc_testing.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b(gc_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["gc_exclusive_scan", "gc_select_if", "gc_partition", "gc_split_radix",
                 "gc_select_if_atomic", "gc_select_if_atomic_tile", "gc_workspace_bytes", "gc_query_device_status",
                 "gc_status_string", "gc_workspace_init", "gc_tile_elements",
                 "gc_testing_select_if_skip_tile0", "gc_inclusive_scan", "gc_select_if_pred",
                 "gc_partition_pred", "gc_select_if_noalloc", "gc_radix_sort",
                 "gc_testing_exclusive_scan_stalled_barrier"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(gc.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code in range(8):
        s = lib.gc_status_string(code)
        assert s and s.decode().startswith(gc.STATUS[code])
    assert lib.gc_status_string(99) == b"unknown gc_status"
    assert b"sm_103a" in lib.gc_version()


def test_workspace_sizes(lib):
    for op in range(5):
        assert lib.gc_workspace_bytes(op, 0, gc.I32) >= 512
        assert lib.gc_workspace_bytes(op, 2 ** 31, gc.I32) == 0
        assert lib.gc_tile_elements(op) >= 2048
    assert lib.gc_workspace_bytes(9, 100, gc.I32) == 0
    assert lib.gc_workspace_bytes(gc.OP_EXCLUSIVE_SCAN, 100, 7) == 0
    # float scan keeps a double prefix per tile beside the status words
    n = 1 << 20
    assert lib.gc_workspace_bytes(gc.OP_EXCLUSIVE_SCAN, n, gc.F32) > \
        lib.gc_workspace_bytes(gc.OP_EXCLUSIVE_SCAN, n, gc.I32)
    # radix holds the ping-pong keys and payloads: at least 8 bytes per element
    assert lib.gc_workspace_bytes(gc.OP_SPLIT_RADIX, n, gc.U32) >= 8 * n
    # monotone in n
    sizes = [lib.gc_workspace_bytes(gc.OP_SELECT_IF, k, gc.I32) for k in (1, 10**3, 10**6, 10**9)]
    assert sizes == sorted(sizes)


# Fake device addresses: never dereferenced, every call fails validation first.
IN, OUT, CNT, WS = 0x10000000, 0x20000000, 0x30000000, 0x40000000
BIG = 1 << 28


def sel(lib, *, i=IN, o=OUT, c=CNT, n=1000, dt=gc.I32, p=gc.NONZERO, ws=WS, wsb=BIG,
        fn="gc_select_if"):
    return getattr(lib, fn)(i, o, c, n, dt, p, ws, wsb, None)


@pytest.mark.parametrize("fn", ["gc_select_if", "gc_select_if_atomic", "gc_select_if_atomic_tile",
                                "gc_partition"])
def test_select_like_validation(lib, fn):
    E = {v: k for k, v in gc.STATUS.items()}
    assert sel(lib, fn=fn, n=2 ** 31) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, ws=None) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, ws=WS + 16) == E["GC_ERR_MISALIGNED"]
    assert sel(lib, fn=fn, wsb=100) == E["GC_ERR_WORKSPACE_TOO_SMALL"]
    assert sel(lib, fn=fn, i=None) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, o=None) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, c=None) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, i=IN + 2) == E["GC_ERR_MISALIGNED"]
    assert sel(lib, fn=fn, o=OUT + 1) == E["GC_ERR_MISALIGNED"]
    assert sel(lib, fn=fn, c=CNT + 2) == E["GC_ERR_MISALIGNED"]
    assert sel(lib, fn=fn, dt=gc.F32, p=gc.ODD) == E["GC_ERR_UNSUPPORTED"]
    assert sel(lib, fn=fn, dt=gc.F32, p=gc.EVEN) == E["GC_ERR_UNSUPPORTED"]
    assert sel(lib, fn=fn, p=7) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, dt=5) == E["GC_ERR_INVALID_VALUE"]
    assert sel(lib, fn=fn, o=IN + 400) == E["GC_ERR_INVALID_VALUE"]        # in/out overlap
    assert sel(lib, fn=fn, c=OUT + 40) == E["GC_ERR_INVALID_VALUE"]        # count inside out
    assert sel(lib, fn=fn, i=WS + 4096) == E["GC_ERR_INVALID_VALUE"]       # input inside workspace


def test_scan_validation(lib):
    E = {v: k for k, v in gc.STATUS.items()}
    f = lib.gc_exclusive_scan
    assert f(IN, OUT, None, 2 ** 31, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, IN + 8, None, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]  # partial overlap
    assert f(IN, OUT, OUT + 12, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]  # total in out
    assert f(IN, OUT, CNT + 1, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_MISALIGNED"]
    assert f(IN, OUT, None, 1000, 3, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, OUT, None, 1000, gc.F32, WS, 530, None) == E["GC_ERR_WORKSPACE_TOO_SMALL"]
    assert f(None, OUT, None, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]


def test_stalled_barrier_hook_validation(lib):
    # Refused before any CUDA call: the hook needs the persistent kernel's
    # path (a 16-byte-aligned input) and at least one element.
    E = {v: k for k, v in gc.STATUS.items()}
    f = lib.gc_testing_exclusive_scan_stalled_barrier
    assert f(IN, OUT, None, 0, gc.I32, WS, BIG, 1000, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN + 4, OUT, None, 1000, gc.I32, WS, BIG, 1000, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, OUT, None, 1000, gc.I32, WS + 8, BIG, 1000, None) == E["GC_ERR_MISALIGNED"]


def test_pred_validation(lib):
    E = {v: k for k, v in gc.STATUS.items()}
    good = gc.Predicate(gc.LT, 5, 0)
    for fn in (lib.gc_select_if_pred, lib.gc_partition_pred):
        assert fn(IN, OUT, CNT, 1000, gc.I32, None, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
        bad = gc.Predicate(8, 0, 0)
        assert fn(IN, OUT, CNT, 1000, gc.I32, bad, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
        bad = gc.Predicate(-1, 0, 0)
        assert fn(IN, OUT, CNT, 1000, gc.I32, bad, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
        # float32 accepts every comparison (unlike ODD/EVEN); the other checks still apply
        assert fn(IN + 2, OUT, CNT, 1000, gc.F32, good, WS, BIG, None) == E["GC_ERR_MISALIGNED"]
        assert fn(IN, OUT, CNT, 1000, gc.F32, good, WS, 100, None) == E["GC_ERR_WORKSPACE_TOO_SMALL"]
        assert fn(IN, IN + 40, CNT, 1000, gc.I32, good, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    f = lib.gc_inclusive_scan
    assert f(IN, IN + 8, None, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, OUT, None, 2 ** 31, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert lib.gc_workspace_bytes(gc.OP_INCLUSIVE_SCAN, 1 << 20, gc.F32) == \
        lib.gc_workspace_bytes(gc.OP_EXCLUSIVE_SCAN, 1 << 20, gc.F32)


def test_predicate_helper_bits():
    import torch
    x = torch.zeros(1, dtype=torch.float32)
    p = gc.predicate(x, "<", 2.5)
    assert p.cmp == gc.LT and p.operand == 0x40200000
    p = gc.predicate(torch.zeros(1, dtype=torch.int32), ">=", -1)
    assert p.operand == 0xFFFFFFFF
    p = gc.predicate(x, "mask!=", 0, 1)
    assert (p.cmp, p.operand, p.mask) == (gc.MASK_NE, 0, 1)


def test_radix_validation(lib):
    E = {v: k for k, v in gc.STATUS.items()}
    f = lib.gc_split_radix
    K2, V1, V2 = 0x50000000, 0x60000000, 0x70000000
    ok = dict(ki=IN, vi=V1, ko=K2, vo=V2, n=1000, b=0, e=32, ws=WS, wsb=BIG)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["ki"], a["vi"], a["ko"], a["vo"], a["n"], a["b"], a["e"], a["ws"], a["wsb"], None)
    assert call(b=-1) == E["GC_ERR_INVALID_VALUE"]
    assert call(e=33) == E["GC_ERR_INVALID_VALUE"]
    assert call(b=9, e=8) == E["GC_ERR_INVALID_VALUE"]
    assert call(vi=None) == E["GC_ERR_INVALID_VALUE"]
    assert call(vo=None) == E["GC_ERR_INVALID_VALUE"]
    assert call(vo=IN + 64) == E["GC_ERR_INVALID_VALUE"]       # payload over keys
    assert call(ko=IN + 8) == E["GC_ERR_INVALID_VALUE"]        # keys partially overlap
    assert call(vi=V1 + 2) == E["GC_ERR_MISALIGNED"]
    assert call(wsb=1 << 12) == E["GC_ERR_WORKSPACE_TOO_SMALL"]
    assert call(n=2 ** 31) == E["GC_ERR_INVALID_VALUE"]


def test_radix_sort_validation(lib):
    E = {v: k for k, v in gc.STATUS.items()}
    f = lib.gc_radix_sort
    K2, V1, V2 = 0x50000000, 0x60000000, 0x70000000
    ok = dict(ki=IN, vi=V1, ko=K2, vo=V2, n=1000, dt=gc.F32, ws=WS, wsb=BIG)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["ki"], a["vi"], a["ko"], a["vo"], a["n"], a["dt"], a["ws"], a["wsb"], None)
    assert call(dt=3) == E["GC_ERR_INVALID_VALUE"]
    assert call(dt=-1) == E["GC_ERR_INVALID_VALUE"]
    assert call(vi=None) == E["GC_ERR_INVALID_VALUE"]
    assert call(vo=None) == E["GC_ERR_INVALID_VALUE"]
    assert call(vo=IN + 64) == E["GC_ERR_INVALID_VALUE"]
    assert call(ko=IN + 8) == E["GC_ERR_INVALID_VALUE"]
    assert call(ki=IN + 2) == E["GC_ERR_MISALIGNED"]
    assert call(vi=V1 + 2) == E["GC_ERR_MISALIGNED"]
    assert call(wsb=1 << 12) == E["GC_ERR_WORKSPACE_TOO_SMALL"]
    assert call(n=2 ** 31) == E["GC_ERR_INVALID_VALUE"]
    assert call(ws=None) == E["GC_ERR_INVALID_VALUE"]
    for dt in (gc.I32, gc.U32, gc.F32):
        # the ping-pong buffers of the split sort plus a 256-word count per 4096-key tile
        for n in (1, 4096, 12345, 1 << 28):
            got = lib.gc_workspace_bytes(gc.OP_RADIX_SORT, n, dt)
            table = -(-4 * 256 * -(-n // 4096) // 256) * 256
            assert got == lib.gc_workspace_bytes(gc.OP_SPLIT_RADIX, n, gc.U32) + table, n
    assert lib.gc_workspace_bytes(gc.OP_RADIX_SORT, 12345, 7) == 0
    assert lib.gc_tile_elements(gc.OP_RADIX_SORT) == 4096


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.arange(10, dtype=torch.int32)
    with pytest.raises(ValueError):
        gc.exclusive_scan(x, out=x.clone(), ws=torch.zeros(4096, dtype=torch.uint8))
    with pytest.raises(TypeError):
        gc.dtype_code(torch.zeros(3, dtype=torch.int64))


def test_shard_entry_point_validation(lib):
    """The sharded entry points reject bad arguments on the host."""
    import ctypes
    E = {v: k for k, v in gc.STATUS.items()}
    V = ctypes.c_void_p
    f = lib.gc_reduce
    f.argtypes = [V, V, ctypes.c_size_t, ctypes.c_int, V, ctypes.c_size_t, V]
    assert f(IN, None, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, CNT + 2, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_MISALIGNED"]
    assert f(IN, IN + 40, 1000, gc.I32, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]  # total in input
    assert f(IN, CNT, 1000, 9, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    f = lib.gc_count_if
    f.argtypes = [V, V, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, V, ctypes.c_size_t, V]
    assert f(IN, CNT, 1000, gc.F32, gc.ODD, WS, BIG, None) == E["GC_ERR_UNSUPPORTED"]
    assert f(IN, None, 1000, gc.I32, gc.ODD, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    f = lib.gc_exclusive_scan_carry
    f.argtypes = [V, V, V, ctypes.c_size_t, ctypes.c_int, V, V, ctypes.c_size_t, V]
    assert f(IN, OUT, None, 1000, gc.I32, None, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, OUT, None, 1000, gc.I32, CNT + 1, WS, BIG, None) == E["GC_ERR_MISALIGNED"]
    assert f(IN, OUT, None, 1000, gc.I32, OUT + 8, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    f = lib.gc_select_if_at
    f.argtypes = [V, V, ctypes.c_size_t, V, V, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, V,
                  ctypes.c_size_t, V]
    assert f(IN, OUT, 5000, None, CNT, 1000, gc.I32, gc.ODD, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, OUT, 5000, CNT + 4, CNT, 1000, gc.I32, gc.ODD, WS, BIG, None) == E["GC_ERR_MISALIGNED"]
    assert f(IN, OUT, 0, CNT + 8, CNT, 1000, gc.I32, gc.ODD, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    # the whole output (capacity) must not overlap the input
    assert f(IN, IN - 4 * 100, 5000, CNT + 8, CNT, 1000, gc.I32, gc.ODD, WS, BIG, None) == \
        E["GC_ERR_INVALID_VALUE"]
    f = lib.gc_partition_at
    f.argtypes = [V, V, ctypes.c_size_t, V, V, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, V,
                  ctypes.c_size_t, V]
    assert f(IN, OUT, 999, CNT + 8, CNT, 1000, gc.I32, gc.ODD, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(IN, OUT, 5000, None, CNT, 1000, gc.I32, gc.ODD, WS, BIG, None) == E["GC_ERR_INVALID_VALUE"]
    f = lib.gc_shard_offsets
    U64P = ctypes.POINTER(ctypes.c_uint64)
    f.argtypes = [ctypes.c_int, ctypes.c_int, V, U64P, ctypes.c_size_t, ctypes.c_size_t, V, V]
    sizes = (ctypes.c_uint64 * 4)(1, 2, 3, 4)
    assert f(gc.OP_SELECT_IF, gc.U32, CNT, None, 4, 4, OUT, None) == E["GC_ERR_INVALID_VALUE"]   # rank >= parts
    assert f(gc.OP_SELECT_IF, gc.U32, CNT, None, 0, 0, OUT, None) == E["GC_ERR_INVALID_VALUE"]   # no parts
    assert f(gc.OP_PARTITION, gc.U32, CNT, None, 4, 1, OUT, None) == E["GC_ERR_INVALID_VALUE"]   # sizes needed
    assert f(gc.OP_RADIX_SORT, gc.U32, CNT, sizes, 4, 1, OUT, None) == E["GC_ERR_INVALID_VALUE"]
    assert f(gc.OP_SELECT_IF, gc.U32, CNT, None, 4, 1, OUT + 4, None) == E["GC_ERR_MISALIGNED"]
    big = (ctypes.c_uint64 * 2)(1, 1 << 31)
    assert f(gc.OP_PARTITION, gc.U32, CNT, big, 2, 1, OUT, None) == E["GC_ERR_INVALID_VALUE"]
    for op in (gc.OP_REDUCE, gc.OP_COUNT_IF):
        assert lib.gc_workspace_bytes(op, 1 << 20, gc.I32) >= 512
