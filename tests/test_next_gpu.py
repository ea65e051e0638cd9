"""Parity of the widened entry points with the oracle, on the GPU through the C ABI:
the inclusive scan, select-if / partition with parameterised predicates
(every comparison in every dtype's order, and masked-bit tests), and the
typed 8-bit-digit radix sort.

Same bar as the core path: integer results bit-exact, float32 scans within
1e-5 relative of the float64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import dev, empty_like_offset, f32_within, host
from partition_pass_tile_gb300 import gc, synth

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(77)
NP = {gc.I32: np.int32, gc.U32: np.uint32, gc.F32: np.float32}


def sizes(op):
    T = gc.tile_elements(op)
    return [1, 2, 5, 33, 129, T - 1, T, T + 1, 3 * T + 17, 100_003]


# ---------------------------------------------------------------- inclusive scan

@pytest.mark.parametrize("dt", [gc.I32, gc.U32, gc.F32])
@pytest.mark.parametrize("offset", [0, 1])
def test_inclusive_scan_sizes(orc, dt, offset):
    for n in sizes(gc.OP_INCLUSIVE_SCAN):
        if dt == gc.F32:
            x = synth.scan_unit_f32(n, int(RNG.integers(1 << 30)))
        else:
            x = synth.uniform_u32(n, int(RNG.integers(1 << 30))).view(NP[dt])
        want, wt = orc.inclusive_scan(x)
        xd = dev(x, offset)
        out, tot = gc.inclusive_scan(xd, out=empty_like_offset(xd, offset))
        got = host(out)
        if dt == gc.F32:
            bad, worst = f32_within(got, want)
            assert bad.size == 0, (n, bad[:5], worst)
        else:
            assert np.array_equal(got, want), (n, np.flatnonzero(got != want)[:5])
            assert host(tot)[0] == wt


def test_inclusive_scan_closed_form_and_in_place(orc):
    n = synth.SIZES["scan"]
    x = synth.scan_mod8(n)
    xd = dev(x)
    gc.inclusive_scan(xd, out=xd)  # in place
    i = np.arange(n, dtype=np.int64)
    r = i % 8
    want = 36 * (i // 8) + (r + 1) * (r + 2) // 2  # (i%8)+1 summed through i
    assert np.array_equal(host(xd).astype(np.int64), want)
    xf = synth.every_fourth_two_f32(n)
    out, tot = gc.inclusive_scan(dev(xf))
    assert np.array_equal(host(out).astype(np.float64), (i + 1 + (i + 4) // 4).astype(np.float64))
    assert float(host(tot)[0]) == 12_500_000


# ---------------------------------------------------------------- parameterised predicates

def pred_input(n, dt):
    if dt == gc.I32:
        x = RNG.integers(-40, 41, size=n).astype(np.int32)
        x[::23] = np.iinfo(np.int32).min
        x[7::29] = np.iinfo(np.int32).max
    elif dt == gc.U32:
        x = RNG.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
        x[::11] = 9
    else:
        x = (RNG.standard_normal(n) * 2).astype(np.float32)
        sp = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1e-45, -1e-45, 1.5], np.float32)
        x[:: 5] = sp[RNG.integers(0, 8, size=x[::5].shape[0])]
    return x


OPERANDS = {gc.I32: [0, -7, 2147483647, -2147483648],
            gc.U32: [9, 2 ** 31, 0, 2 ** 32 - 1],
            gc.F32: [0.0, -0.0, 1.5, float("nan"), float("inf"), float("-inf"), -1e-45]}
MASKS = [(1, 0), (1, 1), (0x80000000, 0), (0xF0, 0x50)]


def _cases(dt):
    for v in OPERANDS[dt]:
        for cmp in (gc.LT, gc.LE, gc.GT, gc.GE, gc.EQ, gc.NE):
            yield cmp, v, 0
    for mask, v in MASKS:
        yield gc.MASK_EQ, v, mask
        yield gc.MASK_NE, v, mask


@pytest.mark.parametrize("dt", [gc.I32, gc.U32, gc.F32])
@pytest.mark.parametrize("offset", [0, 3])
def test_select_if_pred(orc, dt, offset):
    for n in (1, 33, gc.tile_elements(gc.OP_SELECT_IF) + 1, 70_001):
        x = pred_input(n, dt)
        xd = dev(x, offset)
        for cmp, v, mask in _cases(dt):
            want = orc.select_if_cmp(x, cmp, v, mask)
            out = empty_like_offset(xd, (offset + 1) % 4, fill=-3)
            out, cnt = gc.select_if_pred(xd, gc.predicate(xd, cmp, v, mask), out=out)
            m = int(host(cnt)[0])
            assert m == want.shape[0], (n, cmp, v, mask)
            assert np.array_equal(host(out)[:m].view(np.uint32), want.view(np.uint32)), (n, cmp, v)


@pytest.mark.parametrize("dt", [gc.I32, gc.U32, gc.F32])
def test_partition_pred(orc, dt):
    for n in (1, 33, gc.tile_elements(gc.OP_PARTITION) + 1, 70_001):
        x = pred_input(n, dt)
        xd = dev(x)
        for cmp, v, mask in _cases(dt):
            want, t = orc.partition_cmp(x, cmp, v, mask)
            out, ct = gc.partition_pred(xd, gc.predicate(xd, cmp, v, mask))
            assert int(host(ct)[0]) == t, (n, cmp, v, mask)
            assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32)), (n, cmp, v)


def test_pred_at_scale(orc):
    """2^26 elements: a float range cut and an int32 partition, every element compared."""
    n = 1 << 26
    xf = synth.scan_unit_f32(n, 31)
    want = orc.select_if_cmp(xf, O.GT, 0.75)
    out, cnt = gc.select_if_pred(dev(xf), gc.predicate(torch.zeros(1), ">", 0.75))
    m = int(host(cnt)[0])
    assert m == want.shape[0] and np.array_equal(host(out)[:m], want)
    xi = synth.uniform_i32(n, 32)
    want, t = orc.partition_cmp(xi, O.LT, -(2 ** 30))
    out, ct = gc.partition_pred(dev(xi), gc.predicate(torch.zeros(1, dtype=torch.int32), "<", -(2 ** 30)))
    assert int(host(ct)[0]) == t and np.array_equal(host(out), want)


# ---------------------------------------------------------------- typed radix sort

def radix_input(n, dt, seed):
    rng = np.random.default_rng(seed)
    if dt == gc.I32:
        x = rng.integers(-2 ** 31, 2 ** 31, size=n, dtype=np.int64).astype(np.int32)
        x[::17] = rng.integers(-3, 4, size=x[::17].shape[0])  # many duplicates around 0
        x[5::31] = np.iinfo(np.int32).min
        x[6::37] = np.iinfo(np.int32).max
    elif dt == gc.U32:
        x = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
        x[::13] = 7
    else:
        x = (rng.standard_normal(n) * 1e3).astype(np.float32)
        sp = np.array([0x00000000, 0x80000000, 0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001,
                       0x7F800000, 0xFF800000, 0x00000001, 0x80000001, 0x3F800000, 0xBF800000],
                      dtype=np.uint32).view(np.float32)
        x[::6] = sp[rng.integers(0, sp.shape[0], size=x[::6].shape[0])]
    return x


@pytest.mark.parametrize("dt", [gc.I32, gc.U32, gc.F32])
@pytest.mark.parametrize("offset,with_vals", [(0, True), (0, False), (1, True)])
def test_radix_sort_sizes(orc, dt, offset, with_vals):
    for n in sizes(gc.OP_RADIX_SORT):
        x = radix_input(n, dt, n + 7 * dt)
        vals = np.arange(n, dtype=np.uint32) if with_vals else None
        wk, wv = orc.radix_sort(x, vals)
        kd = dev(x, offset)
        vd = dev(vals, offset) if with_vals else None
        ko, vo = gc.radix_sort(kd, vd, keys_out=empty_like_offset(kd, offset),
                               vals_out=empty_like_offset(vd, offset) if with_vals else None)
        assert np.array_equal(host(ko).view(np.uint32), wk.view(np.uint32)), (n, dt)
        if with_vals:
            assert np.array_equal(host(vo), wv), (n, dt)


@pytest.mark.parametrize("dt", [gc.I32, gc.F32])
def test_radix_sort_in_place_and_order(orc, dt):
    n = 3 * gc.tile_elements(gc.OP_RADIX_SORT) + 5
    x = radix_input(n, dt, 99)
    vals = np.arange(n, dtype=np.uint32)
    kd, vd = dev(x), dev(vals)
    gc.radix_sort(kd, vd, keys_out=kd, vals_out=vd)  # in place
    wk, wv = orc.radix_sort(x, vals)
    got_k, got_v = host(kd), host(vd)
    assert np.array_equal(got_k.view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(got_v, wv)
    assert np.array_equal(x[got_v].view(np.uint32), got_k.view(np.uint32))
    if dt == gc.I32:
        assert np.all(got_k[1:] >= got_k[:-1])
    else:
        finite = got_k[~np.isnan(got_k)]
        assert np.all(finite[1:] >= finite[:-1])


def test_radix_sort_float_at_scale(orc):
    """2^26 float32 keys (normal, with specials), index payload: every element compared."""
    n = 1 << 26
    x = radix_input(n, gc.F32, 2026)
    vals = np.arange(n, dtype=np.uint32)
    wk, wv = orc.radix_sort(x, vals)
    ko, vo = gc.radix_sort(dev(x), dev(vals))
    assert np.array_equal(host(ko).view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(host(vo), wv)


def test_radix_sort_duplicates_and_uint32_at_scale(orc):
    """2^25 int32 keys drawn from 1000 values (long runs of equal keys: stability
    across tiles and passes), and 2^25 uint32 keys against the one-bit oracle."""
    n = 1 << 25
    rng = np.random.default_rng(4242)
    x = (rng.integers(-500, 500, size=n)).astype(np.int32)
    vals = np.arange(n, dtype=np.uint32)
    wk, wv = orc.radix_sort(x, vals)
    ko, vo = gc.radix_sort(dev(x), dev(vals))
    assert np.array_equal(host(ko), wk)
    assert np.array_equal(host(vo), wv)
    ku, _ = synth.radix_keys(n, 77)
    wk, wv = orc.split_radix(ku, vals)
    ko, vo = gc.radix_sort(dev(ku), dev(vals))
    assert np.array_equal(host(ko), wk) and np.array_equal(host(vo), wv)
