"""Plain CPU oracle for the predicate -> exclusive scan -> scatter path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library under ``partition_pass_tile_gb300``
never imports it, and this package imports nothing from that library.

The arithmetic lives in ``oracle.c`` (single-threaded C, one sequential loop
per definition); this module only compiles it with gcc, loads it with ctypes
and moves numpy arrays in and out.  Citations for every definition are in the
C source.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):

* exclusive_scan (int32/uint32): printed worked example (CIS 565 scan test
  log), closed forms for the (i % 8) + 1 and every-fourth-is-2 inputs,
  first-difference invariant, brute force.
* exclusive_scan (float32 -> float64): exact integer prefix of inputs that are
  multiples of 2^-24, closed form for the every-fourth-is-2 input.
* inclusive_scan (int32/uint32, float32 -> float64): the identity
  inclusive[i] = exclusive[i] + in[i] against the exclusive forms above, with
  equal totals; storing an element before adding it fails it.
* select_if / count_if: printed worked example (CIS 565 compaction log),
  O(n^2) brute-force rank counting, subsequence invariant, all/none kept.
* partition: brute-force ranks for both halves, permutation + stability
  invariants, the i - rank[i] identity.
* split_radix: numpy's stable argsort (a library routine) on keys, payload
  permutation, single-bit case against partition.
* radix_sort (typed keys): numpy's stable argsort on int32 / float32 keys
  without NaN or -0.0, a hand-written totalOrder sequence of float special
  values, and split_radix for uint32.
* select_if_cmp / partition_cmp: numpy's element-wise comparisons and
  masked-bit tests (library routines, IEEE semantics for float32) on inputs
  with every float special value; the fixed predicates as special cases.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

I32, U32, F32 = 0, 1, 2
NONZERO, ODD, EVEN = 0, 1, 2
LT, LE, GT, GE, EQ, NE, MASK_EQ, MASK_NE = range(8)

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"

_lib = None


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math).

    -O2 without -ffast-math keeps every floating-point add in source order.
    """
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
             "-fno-fast-math", "-o", str(tmp), str(_SRC)],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str | os.PathLike | None = None) -> ctypes.CDLL:
    """Load a compiled oracle (the default one, or another build of oracle.c)."""
    lib = ctypes.CDLL(str(path if path is not None else build()))
    P = ctypes.c_void_p
    Z = ctypes.c_size_t
    I = ctypes.c_int
    lib.orc_pred_supported.argtypes = [I, I]
    lib.orc_pred_supported.restype = I
    lib.orc_count_if.argtypes = [P, Z, I, I]
    lib.orc_count_if.restype = Z
    lib.orc_exclusive_scan_u32.argtypes = [P, P, Z]
    lib.orc_exclusive_scan_u32.restype = ctypes.c_uint32
    lib.orc_exclusive_scan_f32.argtypes = [P, P, Z]
    lib.orc_exclusive_scan_f32.restype = ctypes.c_double
    lib.orc_inclusive_scan_u32.argtypes = [P, P, Z]
    lib.orc_inclusive_scan_u32.restype = ctypes.c_uint32
    lib.orc_inclusive_scan_f32.argtypes = [P, P, Z]
    lib.orc_inclusive_scan_f32.restype = ctypes.c_double
    lib.orc_select_if.argtypes = [P, P, Z, I, I]
    lib.orc_select_if.restype = Z
    lib.orc_partition.argtypes = [P, P, Z, I, I]
    lib.orc_partition.restype = Z
    lib.orc_split_radix.argtypes = [P, P, P, P, Z, I, I]
    lib.orc_split_radix.restype = I
    U = ctypes.c_uint32
    lib.orc_select_if_cmp.argtypes = [P, P, Z, I, I, U, U]
    lib.orc_select_if_cmp.restype = Z
    lib.orc_partition_cmp.argtypes = [P, P, Z, I, I, U, U]
    lib.orc_partition_cmp.restype = Z
    lib.orc_radix_sort.argtypes = [P, P, P, P, Z, I]
    lib.orc_radix_sort.restype = I
    lib.orc_count_out_of_order.argtypes = [P, P, Z]
    lib.orc_count_out_of_order.restype = Z
    return lib


def _default():
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.int32:
        return I32
    if a.dtype == np.uint32:
        return U32
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle handles int32, uint32 and float32, not {a.dtype}")


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """numpy-facing wrapper around one loaded build of oracle.c."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else _default()

    def pred_supported(self, dtype: int, pred: int) -> bool:
        return bool(self.lib.orc_pred_supported(dtype, pred))

    def exclusive_scan(self, x: np.ndarray):
        """int32/uint32 -> (same dtype, wrapped mod 2^32, total);
        float32 -> (float64 prefixes, float64 total)."""
        x = _c(x)
        if x.dtype == np.float32:
            out = np.empty(x.shape[0], dtype=np.float64)
            tot = self.lib.orc_exclusive_scan_f32(_ptr(x), _ptr(out), x.shape[0])
            return out, float(tot)
        _dtype_code(x)
        out = np.empty_like(x)
        tot = self.lib.orc_exclusive_scan_u32(_ptr(x), _ptr(out), x.shape[0])
        return out, np.array(tot, dtype=np.uint32).view(x.dtype)[()]

    def inclusive_scan(self, x: np.ndarray):
        x = _c(x)
        if x.dtype == np.float32:
            out = np.empty(x.shape[0], dtype=np.float64)
            tot = self.lib.orc_inclusive_scan_f32(_ptr(x), _ptr(out), x.shape[0])
            return out, float(tot)
        _dtype_code(x)
        out = np.empty_like(x)
        tot = self.lib.orc_inclusive_scan_u32(_ptr(x), _ptr(out), x.shape[0])
        return out, np.array(tot, dtype=np.uint32).view(x.dtype)[()]

    def count_if(self, x: np.ndarray, pred: int) -> int:
        x = _c(x)
        return int(self.lib.orc_count_if(_ptr(x), x.shape[0], _dtype_code(x), pred))

    def select_if(self, x: np.ndarray, pred: int) -> np.ndarray:
        x = _c(x)
        out = np.empty_like(x)
        m = self.lib.orc_select_if(_ptr(x), _ptr(out), x.shape[0], _dtype_code(x), pred)
        return out[:m].copy()

    def partition(self, x: np.ndarray, pred: int):
        """-> (partitioned array, size of the predicate-true half)."""
        x = _c(x)
        out = np.empty_like(x)
        t = self.lib.orc_partition(_ptr(x), _ptr(out), x.shape[0], _dtype_code(x), pred)
        return out, int(t)

    @staticmethod
    def operand_bits(x: np.ndarray, value) -> int:
        """The 32-bit pattern of `value` in x's dtype."""
        return int(np.array([value], dtype=x.dtype).view(np.uint32)[0])

    def select_if_cmp(self, x: np.ndarray, cmp: int, value=0, mask: int = 0) -> np.ndarray:
        """value: a number of x's dtype for LT..NE, a raw 32-bit pattern for MASK_*."""
        x = _c(x)
        out = np.empty_like(x)
        v = int(value) & 0xFFFFFFFF if cmp >= MASK_EQ else self.operand_bits(x, value)
        m = self.lib.orc_select_if_cmp(_ptr(x), _ptr(out), x.shape[0], _dtype_code(x), cmp, v,
                                       mask & 0xFFFFFFFF)
        return out[:m].copy()

    def partition_cmp(self, x: np.ndarray, cmp: int, value=0, mask: int = 0):
        x = _c(x)
        out = np.empty_like(x)
        v = int(value) & 0xFFFFFFFF if cmp >= MASK_EQ else self.operand_bits(x, value)
        t = self.lib.orc_partition_cmp(_ptr(x), _ptr(out), x.shape[0], _dtype_code(x), cmp, v,
                                       mask & 0xFFFFFFFF)
        return out, int(t)

    def split_radix(self, keys: np.ndarray, vals: np.ndarray | None = None,
                    begin_bit: int = 0, end_bit: int = 32):
        """-> (keys_out, vals_out or None)."""
        keys = _c(keys.astype(np.uint32, copy=False))
        ko = np.empty_like(keys)
        if vals is not None:
            vals = _c(vals.astype(np.uint32, copy=False))
            vo = np.empty_like(vals)
            rc = self.lib.orc_split_radix(_ptr(keys), _ptr(vals), _ptr(ko), _ptr(vo),
                                          keys.shape[0], begin_bit, end_bit)
        else:
            vo = None
            rc = self.lib.orc_split_radix(_ptr(keys), None, _ptr(ko), None,
                                          keys.shape[0], begin_bit, end_bit)
        if rc != 0:
            raise ValueError("orc_split_radix rejected its arguments")
        return ko, vo

    def radix_sort(self, keys: np.ndarray, vals: np.ndarray | None = None):
        """Stable ascending sort in keys' dtype order (float32: IEEE totalOrder)."""
        keys = _c(keys)
        dt = _dtype_code(keys)
        ko = np.empty_like(keys)
        if vals is not None:
            vals = _c(vals.astype(np.uint32, copy=False))
            vo = np.empty_like(vals)
            rc = self.lib.orc_radix_sort(_ptr(keys), _ptr(vals), _ptr(ko), _ptr(vo), keys.shape[0], dt)
        else:
            vo = None
            rc = self.lib.orc_radix_sort(_ptr(keys), None, _ptr(ko), None, keys.shape[0], dt)
        if rc != 0:
            raise ValueError("orc_radix_sort rejected its arguments")
        return ko, vo

    def count_out_of_order(self, got: np.ndarray, want: np.ndarray) -> int:
        got = _c(got).view(np.uint32)
        want = _c(want).view(np.uint32)
        assert got.shape == want.shape
        return int(self.lib.orc_count_out_of_order(_ptr(got), _ptr(want), got.shape[0]))


def default() -> Oracle:
    return Oracle()
