"""Python binding of libgc (include/gc.h): argument marshalling only.

Every function here turns torch tensors into device pointers, sizes and enum
codes, calls the C entry point of the same name, and raises ``GcError`` on a
non-zero status.  No step of the computation runs in Python: the predicate,
the scan and the scatter all run in libgc's CUDA kernels.  PyTorch supplies
device memory and streams.

The library is loaded on first use from this package's directory; if it has
not been built (``__graft_entry__.build()`` or ``python -m
partition_pass_tile_gb300.build``) the first call raises.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "libgc.so"

# enum values of include/gc.h
I32, U32, F32 = 0, 1, 2
NONZERO, ODD, EVEN = 0, 1, 2
OP_EXCLUSIVE_SCAN, OP_SELECT_IF, OP_PARTITION, OP_SPLIT_RADIX, OP_SELECT_IF_ATOMIC = range(5)
OP_INCLUSIVE_SCAN = 5
OP_RADIX_SORT = 6
OP_REDUCE = 7
OP_COUNT_IF = 8
LT, LE, GT, GE, EQ, NE, MASK_EQ, MASK_NE = range(8)
CMP_NAMES = {"<": LT, "<=": LE, ">": GT, ">=": GE, "==": EQ, "!=": NE,
             "mask==": MASK_EQ, "mask!=": MASK_NE}


class Predicate(ctypes.Structure):
    """gc_predicate: x OP operand in the dtype's order, or (bits & mask) OP operand."""
    _fields_ = [("cmp", ctypes.c_int), ("operand", ctypes.c_uint32), ("mask", ctypes.c_uint32)]
STATUS = {0: "GC_OK", 1: "GC_ERR_INVALID_VALUE", 2: "GC_ERR_UNSUPPORTED",
          3: "GC_ERR_WORKSPACE_TOO_SMALL", 4: "GC_ERR_MISALIGNED", 5: "GC_ERR_CUDA",
          6: "GC_ERR_TIMEOUT", 7: "GC_ERR_DEVICE_CHECK"}
PRED_NAMES = {"nonzero": NONZERO, "odd": ODD, "even": EVEN}

_lib = None


class GcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def load(path: str | Path | None = None) -> ctypes.CDLL:
    """Load libgc.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(python -m partition_pass_tile_gb300.build)")
    lib = ctypes.CDLL(str(p))
    V, Z, I, U64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
    S = ctypes.c_int
    sig = {
        "gc_status_string": ([S], ctypes.c_char_p),
        "gc_version": ([], ctypes.c_char_p),
        "gc_workspace_bytes": ([I, Z, I], Z),
        "gc_tile_elements": ([I], Z),
        "gc_workspace_init": ([V, Z, V], S),
        "gc_exclusive_scan": ([V, V, V, Z, I, V, Z, V], S),
        "gc_select_if": ([V, V, V, Z, I, I, V, Z, V], S),
        "gc_partition": ([V, V, V, Z, I, I, V, Z, V], S),
        "gc_split_radix": ([V, V, V, V, Z, I, I, V, Z, V], S),
        "gc_select_if_atomic": ([V, V, V, Z, I, I, V, Z, V], S),
        "gc_select_if_atomic_tile": ([V, V, V, Z, I, I, V, Z, V], S),
        "gc_query_device_status": ([V, V], S),
        "gc_testing_select_if_skip_tile0": ([V, V, V, Z, I, I, V, Z, U64, V], S),
        "gc_testing_exclusive_scan_stalled_barrier": ([V, V, V, Z, I, V, Z, U64, V], S),
        "gc_inclusive_scan": ([V, V, V, Z, I, V, Z, V], S),
        "gc_select_if_pred": ([V, V, V, Z, I, ctypes.POINTER(Predicate), V, Z, V], S),
        "gc_partition_pred": ([V, V, V, Z, I, ctypes.POINTER(Predicate), V, Z, V], S),
        "gc_radix_sort": ([V, V, V, V, Z, I, V, Z, V], S),
        "gc_reduce": ([V, V, Z, I, V, Z, V], S),
        "gc_count_if": ([V, V, Z, I, I, V, Z, V], S),
        "gc_shard_offsets": ([I, I, V, ctypes.POINTER(U64), Z, Z, V, V], S),
        "gc_exclusive_scan_carry": ([V, V, V, Z, I, V, V, Z, V], S),
        "gc_select_if_at": ([V, V, Z, V, V, Z, I, I, V, Z, V], S),
        "gc_partition_at": ([V, V, Z, V, V, Z, I, I, V, Z, V], S),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise GcError(status, what)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.int32:
        return I32
    if t.dtype == torch.uint32:
        return U32
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"libgc handles int32, uint32 and float32 tensors, not {t.dtype}")


def pred_code(pred) -> int:
    return PRED_NAMES[pred] if isinstance(pred, str) else int(pred)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libgc takes CUDA tensors (device pointers)")
    if not t.is_contiguous():
        raise ValueError("libgc takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def tile_elements(op: int) -> int:
    return int(load().gc_tile_elements(op))


def workspace_bytes(op: int, n: int, dtype: int = I32) -> int:
    return int(load().gc_workspace_bytes(op, n, dtype))


def workspace(op: int, n: int, dtype: int = I32, device=None) -> torch.Tensor:
    """A zero-filled workspace for (op, n, dtype) on `device` (torch-allocated)."""
    nbytes = max(workspace_bytes(op, n, dtype), 512)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def _ws(ws, op, n, dtype, device):
    return ws if ws is not None else workspace(op, n, dtype, device)


def exclusive_scan(x: torch.Tensor, out: torch.Tensor | None = None,
                   total: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                   stream=None, with_total: bool = True):
    """-> (out, total); total is a 1-element device tensor of x's dtype (or None)."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if total is None and with_total:
        total = torch.empty(1, dtype=x.dtype, device=x.device)
    ws = _ws(ws, OP_EXCLUSIVE_SCAN, n, dt, x.device)
    _check(load().gc_exclusive_scan(_ptr(x), _ptr(out), _ptr(total), n, dt, _ptr(ws),
                                    ws.numel(), _stream(stream)), "gc_exclusive_scan")
    return out, total


def inclusive_scan(x: torch.Tensor, out: torch.Tensor | None = None,
                   total: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                   stream=None, with_total: bool = True):
    """-> (out, total) with out[i] = x[0] + ... + x[i]."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if total is None and with_total:
        total = torch.empty(1, dtype=x.dtype, device=x.device)
    ws = _ws(ws, OP_INCLUSIVE_SCAN, n, dt, x.device)
    _check(load().gc_inclusive_scan(_ptr(x), _ptr(out), _ptr(total), n, dt, _ptr(ws),
                                    ws.numel(), _stream(stream)), "gc_inclusive_scan")
    return out, total


def predicate(x: torch.Tensor, cmp, operand=0, mask: int = 0) -> Predicate:
    """A gc_predicate for tensor x: cmp in "<", "<=", ">", ">=", "==", "!=" (operand
    a number of x's dtype) or "mask==", "mask!=" (operand, mask: raw 32-bit patterns)."""
    c = CMP_NAMES[cmp] if isinstance(cmp, str) else int(cmp)
    if c >= MASK_EQ:
        bits = int(operand) & 0xFFFFFFFF
    else:
        np_dtype = {torch.int32: "<i4", torch.uint32: "<u4", torch.float32: "<f4"}[x.dtype]
        import numpy as np
        bits = int(np.array([operand], dtype=np_dtype).view(np.uint32)[0])
    return Predicate(c, bits, int(mask) & 0xFFFFFFFF)


def select_if_pred(x: torch.Tensor, pred: Predicate, out: torch.Tensor | None = None,
                   count: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """Stable select-if with a parameterised predicate -> (out, count)."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if count is None:
        count = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_SELECT_IF, n, dt, x.device)
    _check(load().gc_select_if_pred(_ptr(x), _ptr(out), _ptr(count), n, dt, ctypes.byref(pred),
                                    _ptr(ws), ws.numel(), _stream(stream)), "gc_select_if_pred")
    return out, count


def partition_pred(x: torch.Tensor, pred: Predicate, out: torch.Tensor | None = None,
                   count_true: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                   stream=None):
    """Stable partition with a parameterised predicate -> (out, count_true)."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if count_true is None:
        count_true = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_PARTITION, n, dt, x.device)
    _check(load().gc_partition_pred(_ptr(x), _ptr(out), _ptr(count_true), n, dt,
                                    ctypes.byref(pred), _ptr(ws), ws.numel(), _stream(stream)),
           "gc_partition_pred")
    return out, count_true


def select_if(x: torch.Tensor, pred, out: torch.Tensor | None = None,
              count: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """-> (out, count): out has x's size, its first count[0] elements are the survivors."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if count is None:
        count = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_SELECT_IF, n, dt, x.device)
    _check(load().gc_select_if(_ptr(x), _ptr(out), _ptr(count), n, dt, pred_code(pred),
                               _ptr(ws), ws.numel(), _stream(stream)), "gc_select_if")
    return out, count


def select_if_atomic(x: torch.Tensor, pred, out: torch.Tensor | None = None,
                     count: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                     stream=None, per_tile: bool = False):
    """The atomic-counter comparison path -> (out, count): the survivors in an
    order the atomics decide.  One atomic per survivor (gc_select_if_atomic),
    or per tile with per_tile=True (gc_select_if_atomic_tile)."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if count is None:
        count = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_SELECT_IF_ATOMIC, n, dt, x.device)
    name = "gc_select_if_atomic_tile" if per_tile else "gc_select_if_atomic"
    _check(getattr(load(), name)(_ptr(x), _ptr(out), _ptr(count), n, dt, pred_code(pred),
                                 _ptr(ws), ws.numel(), _stream(stream)), name)
    return out, count


def partition(x: torch.Tensor, pred, out: torch.Tensor | None = None,
              count_true: torch.Tensor | None = None, ws: torch.Tensor | None = None,
              stream=None):
    """-> (out, count_true)."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if count_true is None:
        count_true = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_PARTITION, n, dt, x.device)
    _check(load().gc_partition(_ptr(x), _ptr(out), _ptr(count_true), n, dt, pred_code(pred),
                               _ptr(ws), ws.numel(), _stream(stream)), "gc_partition")
    return out, count_true


def split_radix(keys: torch.Tensor, vals: torch.Tensor | None = None, begin_bit: int = 0,
                end_bit: int = 32, keys_out: torch.Tensor | None = None,
                vals_out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                stream=None):
    """-> (keys_out, vals_out).  Keys and payloads are 32-bit (uint32 or int32 bits)."""
    n = keys.numel()
    for t in (keys, vals):
        if t is not None and t.element_size() != 4:
            raise TypeError("split_radix takes 32-bit keys and payloads")
    if keys_out is None:
        keys_out = torch.empty_like(keys)
    if vals is not None and vals_out is None:
        vals_out = torch.empty_like(vals)
    ws = _ws(ws, OP_SPLIT_RADIX, n, U32, keys.device)
    _check(load().gc_split_radix(_ptr(keys), _ptr(vals), _ptr(keys_out), _ptr(vals_out), n,
                                 begin_bit, end_bit, _ptr(ws), ws.numel(), _stream(stream)),
           "gc_split_radix")
    return keys_out, vals_out


def radix_sort(keys: torch.Tensor, vals: torch.Tensor | None = None,
               keys_out: torch.Tensor | None = None, vals_out: torch.Tensor | None = None,
               ws: torch.Tensor | None = None, stream=None):
    """-> (keys_out, vals_out): stable ascending sort in keys' dtype order (float32:
    IEEE 754 totalOrder), 32-bit payloads carried."""
    n = keys.numel()
    dt = dtype_code(keys)
    if vals is not None and vals.element_size() != 4:
        raise TypeError("radix_sort carries 32-bit payloads")
    if keys_out is None:
        keys_out = torch.empty_like(keys)
    if vals is not None and vals_out is None:
        vals_out = torch.empty_like(vals)
    ws = _ws(ws, OP_RADIX_SORT, n, dt, keys.device)
    _check(load().gc_radix_sort(_ptr(keys), _ptr(vals), _ptr(keys_out), _ptr(vals_out), n, dt,
                                _ptr(ws), ws.numel(), _stream(stream)), "gc_radix_sort")
    return keys_out, vals_out


def query_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronous: the workspace's device-side error code (0 = none), then cleared."""
    return int(load().gc_query_device_status(_ptr(ws), _stream(stream)))


def testing_select_if_skip_tile0(x: torch.Tensor, pred, out, count, ws, timeout_ns: int,
                                 stream=None) -> int:
    """Test hook (include/gc_testing.h): returns the launch status."""
    return int(load().gc_testing_select_if_skip_tile0(
        _ptr(x), _ptr(out), _ptr(count), x.numel(), dtype_code(x), pred_code(pred), _ptr(ws),
        ws.numel(), timeout_ns, _stream(stream)))


def testing_force_fallback(on: bool) -> None:
    """Test hook (include/gc_testing.h): one-tile-per-CTA kernels while on."""
    f = load().gc_testing_force_fallback
    f.argtypes = [ctypes.c_int]
    f.restype = None
    f(1 if on else 0)


def testing_exclusive_scan_stalled_barrier(x: torch.Tensor, out, total, ws, timeout_ns: int,
                                           stream=None) -> int:
    """Test hook (include/gc_testing.h): returns the launch status."""
    return int(load().gc_testing_exclusive_scan_stalled_barrier(
        _ptr(x), _ptr(out), _ptr(total), x.numel(), dtype_code(x), _ptr(ws), ws.numel(),
        timeout_ns, _stream(stream)))


NOALLOC_MAX_ELEMENTS = 1 << 28


def select_if_noalloc_status(stream=None) -> int:
    """Synchronous: the no-workspace entry point's device-side error code
    (0 = none) on the current device, then cleared."""
    f = load().gc_select_if_noalloc_status
    f.argtypes = [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return int(f(_stream(stream)))


def testing_select_if_noalloc_stalled_barrier(x: torch.Tensor, pred, out, count, timeout_ns: int,
                                              stream=None) -> int:
    """Test hook (include/gc_testing.h): returns the launch status."""
    f = load().gc_testing_select_if_noalloc_stalled_barrier
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return int(f(_ptr(x), _ptr(out), _ptr(count), x.numel(), dtype_code(x), pred_code(pred),
                 timeout_ns, _stream(stream)))


def select_if_noalloc(x: torch.Tensor, pred, out: torch.Tensor | None = None,
                      count: torch.Tensor | None = None, stream=None):
    """gc_select_if_noalloc: select-if with the library's own fixed scratch
    (no workspace argument, no allocation by the library).  -> (out, count)."""
    lib = load()
    f = lib.gc_select_if_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    if out is None:
        out = torch.empty_like(x)
    if count is None:
        count = torch.empty(1, dtype=torch.uint32, device=x.device)
    _check(f(_ptr(x), _ptr(out), _ptr(count), x.numel(), dtype_code(x), pred_code(pred),
             _stream(stream)), "gc_select_if_noalloc")
    return out, count


# ---------------------------------------------------------------- shards

def reduce(x: torch.Tensor, total: torch.Tensor | None = None, ws: torch.Tensor | None = None,
           stream=None) -> torch.Tensor:
    """gc_reduce: a 1-element device tensor of x's dtype holding sum(x)."""
    n = x.numel()
    dt = dtype_code(x)
    if total is None:
        total = torch.empty(1, dtype=x.dtype, device=x.device)
    ws = _ws(ws, OP_REDUCE, n, dt, x.device)
    _check(load().gc_reduce(_ptr(x), _ptr(total), n, dt, _ptr(ws), ws.numel(), _stream(stream)),
           "gc_reduce")
    return total


def count_if(x: torch.Tensor, pred, count: torch.Tensor | None = None,
             ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gc_count_if: a 1-element uint32 device tensor, how many elements pred keeps."""
    n = x.numel()
    dt = dtype_code(x)
    if count is None:
        count = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_COUNT_IF, n, dt, x.device)
    _check(load().gc_count_if(_ptr(x), _ptr(count), n, dt, pred_code(pred), _ptr(ws), ws.numel(),
                              _stream(stream)), "gc_count_if")
    return count


def shard_offsets(op: int, totals: torch.Tensor, rank: int, sizes=None, dtype: int | None = None,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gc_shard_offsets for shard `rank` of totals.numel() shards.  Returns one
    element of totals' dtype (scan), one 64-bit offset (select-if) or two
    (partition: kept before, first rejected position; `sizes` = the shards'
    element counts, host integers) as an int64 tensor."""
    parts = totals.numel()
    dt = dtype_code(totals) if dtype is None else dtype
    if out is None:
        if op == OP_EXCLUSIVE_SCAN:
            out = torch.empty(1, dtype=totals.dtype, device=totals.device)
        else:
            # uint64 on the device; int64 here (the offsets stay below 2^63)
            out = torch.empty(2 if op == OP_PARTITION else 1, dtype=torch.int64,
                              device=totals.device)
    h = None
    if sizes is not None:
        h = (ctypes.c_uint64 * parts)(*[int(v) for v in sizes])
    _check(load().gc_shard_offsets(op, dt, _ptr(totals), h, parts, rank, _ptr(out),
                                   _stream(stream)), "gc_shard_offsets")
    return out


def exclusive_scan_carry(x: torch.Tensor, carry: torch.Tensor, out: torch.Tensor | None = None,
                         total: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                         stream=None, with_total: bool = True):
    """-> (out, total): out[i] = carry + x[0] + ... + x[i-1], total = carry + sum(x)."""
    n = x.numel()
    dt = dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if total is None and with_total:
        total = torch.empty(1, dtype=x.dtype, device=x.device)
    ws = _ws(ws, OP_EXCLUSIVE_SCAN, n, dt, x.device)
    _check(load().gc_exclusive_scan_carry(_ptr(x), _ptr(out), _ptr(total), n, dt, _ptr(carry),
                                          _ptr(ws), ws.numel(), _stream(stream)),
           "gc_exclusive_scan_carry")
    return out, total


def select_if_at(x: torch.Tensor, pred, out: torch.Tensor, base: torch.Tensor,
                 count: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """Survivors of x to out[base + rank] (out: the whole output; base: a
    1-element uint64 device tensor) -> (out, count of this call)."""
    n = x.numel()
    dt = dtype_code(x)
    if count is None:
        count = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_SELECT_IF, n, dt, x.device)
    _check(load().gc_select_if_at(_ptr(x), _ptr(out), out.numel(), _ptr(base), _ptr(count), n, dt,
                                  pred_code(pred), _ptr(ws), ws.numel(), _stream(stream)),
           "gc_select_if_at")
    return out, count


def partition_at(x: torch.Tensor, pred, out: torch.Tensor, offsets: torch.Tensor,
                 count_true: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                 stream=None):
    """One shard of a partition into the whole output (offsets: the two uint64
    of shard_offsets) -> (out, this shard's kept count)."""
    n = x.numel()
    dt = dtype_code(x)
    if count_true is None:
        count_true = torch.empty(1, dtype=torch.uint32, device=x.device)
    ws = _ws(ws, OP_PARTITION, n, dt, x.device)
    _check(load().gc_partition_at(_ptr(x), _ptr(out), out.numel(), _ptr(offsets), _ptr(count_true),
                                  n, dt, pred_code(pred), _ptr(ws), ws.numel(), _stream(stream)),
           "gc_partition_at")
    return out, count_true
