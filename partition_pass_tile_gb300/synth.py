"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle.

This module holds only random-number generation and the recipes for the
workloads' inputs; it holds none of the method's arithmetic (no predicate,
no scan, no scatter).  It depends on numpy alone, so importing it loads no
CUDA code.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) in counter form,

    x_i = mix(seed + (i + 1) * GAMMA)   (mod 2^64),  GAMMA = 0x9E3779B97F4A7C15

with mix the published 64-bit finaliser (xor-shift 30, multiply, xor-shift 27,
multiply, xor-shift 31).  Counter form means element i depends only on
(seed, i), so any slice can be generated on its own and in parallel.
``hi32``/``lo32`` are the top and bottom 32 bits of x_i.

Workload recipes (sizes are those of the five benchmark configurations):

* remove_zeros(n=1_047_965, seed=1): int32 x_i >> 62, uniform in {0,1,2,3}.
* scan_mod8(n=10_000_000): int32 (i % 8) + 1.
* scan_unit_f32(n=10_000_000, seed=2): float32 (x_i >> 40) * 2^-24, uniform
  on [0, 1) and exactly a multiple of 2^-24.
* every_fourth_two_f32(n): float32, 2.0 where i % 4 == 0 else 1.0 (the Day 32
  scan page's input).
* uniform_i32(n, seed): int32 reinterpretation of hi32 (keep-odd uses seed 3
  and n = 8_387_997; the partition workload uses seed 4 and n = 2^28).
* keep_fraction(n, p, seed): two draws from one x_i; kept iff
  hi32 < round(p * 2^32), and a kept element is lo32 | 1 (never zero), a
  dropped one 0.  Selected with NONZERO.
* radix_keys(n=2^26, seed=5): uint32 hi32 keys with payload i.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

SIZES = {
    "remove_zeros": 1_047_965,        # 2^20 - 611
    "scan": 10_000_000,
    "keep_odd": 8_387_997,            # 2^23 - 611
    "keep_odd_literal": 8_388_597,    # the digit string printed beside it
    "partition": 1 << 28,
    "radix": 1 << 26,
}
SEEDS = {"remove_zeros": 1, "scan_f32": 2, "keep_odd": 3, "partition": 4,
         "radix": 5, "keep_0.01": 41, "keep_0.50": 42, "keep_0.99": 43}


def _mix(z: np.ndarray) -> np.ndarray:
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _chunked(n: int, fill) -> None:
    """Run fill(start, stop) over [0, n) in chunks, on a few threads."""
    starts = list(range(0, n, _CHUNK))
    if len(starts) <= 1:
        for s in starts:
            fill(s, min(n, s + _CHUNK))
        return
    workers = max(1, min(len(starts), os.cpu_count() or 1, 16))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda s: fill(s, min(n, s + _CHUNK)), starts))


def splitmix64(seed: int, start: int, stop: int) -> np.ndarray:
    """x_i for i in [start, stop), as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, stop + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * GAMMA
        return _mix(z)


def hi32(x: np.ndarray) -> np.ndarray:
    return (x >> np.uint64(32)).astype(np.uint32)


def lo32(x: np.ndarray) -> np.ndarray:
    return (x & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def uniform_u32(n: int, seed: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)

    def fill(a, b):
        out[a:b] = hi32(splitmix64(seed, a, b))
    _chunked(n, fill)
    return out


def uniform_i32(n: int, seed: int) -> np.ndarray:
    return uniform_u32(n, seed).view(np.int32)


def remove_zeros(n: int = SIZES["remove_zeros"], seed: int = SEEDS["remove_zeros"]) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)

    def fill(a, b):
        out[a:b] = (splitmix64(seed, a, b) >> np.uint64(62)).astype(np.int32)
    _chunked(n, fill)
    return out


def scan_mod8(n: int = SIZES["scan"]) -> np.ndarray:
    return (np.arange(n, dtype=np.int64) % 8 + 1).astype(np.int32)


def scan_unit_f32(n: int = SIZES["scan"], seed: int = SEEDS["scan_f32"]) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)

    def fill(a, b):
        top24 = (splitmix64(seed, a, b) >> np.uint64(40)).astype(np.float64)
        out[a:b] = (top24 * 2.0 ** -24).astype(np.float32)
    _chunked(n, fill)
    return out


def every_fourth_two_f32(n: int = SIZES["scan"]) -> np.ndarray:
    out = np.ones(n, dtype=np.float32)
    out[0::4] = 2.0
    return out


def keep_threshold(p: float) -> int:
    return min(int(round(p * 2.0 ** 32)), 2 ** 32)


def keep_fraction(n: int, p: float, seed: int) -> np.ndarray:
    thr = keep_threshold(p)
    out = np.empty(n, dtype=np.int32)

    def fill(a, b):
        x = splitmix64(seed, a, b)
        kept = hi32(x).astype(np.uint64) < np.uint64(thr)
        v = lo32(x) | np.uint32(1)
        out[a:b] = np.where(kept, v, np.uint32(0)).view(np.int32)
    _chunked(n, fill)
    return out


def radix_keys(n: int = SIZES["radix"], seed: int = SEEDS["radix"]):
    """-> (uint32 keys, uint32 payload = original index)."""
    return uniform_u32(n, seed), np.arange(n, dtype=np.uint32)
