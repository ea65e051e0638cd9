"""Seeded random sweep over the entry points on the GPU, each case compared
with the oracle: random sizes (including just past tile multiples and the
ragged tails), 4-byte pointer offsets (the scalar kernels), every dtype and
predicate, random comparison operands and masks, radix bit ranges and
payload or not.  Integers bit-exact, float32 scans within 1e-5 relative of
the float64 oracle."""

import numpy as np
import pytest

import oracle as O
from gpu_util import dev, empty_like_offset, f32_within, host
from partition_pass_tile_gb300 import gc

pytestmark = pytest.mark.gpu

NP = {gc.I32: np.int32, gc.U32: np.uint32, gc.F32: np.float32}
CASES = 140


def rand_size(rng, op):
    T = gc.tile_elements(op)
    kind = rng.integers(0, 3)
    if kind == 0:
        return int(rng.integers(1, 4 * T))
    if kind == 1:
        return int(T * rng.integers(1, 40) + rng.integers(-3, 4))
    return int(rng.integers(1, 300_000))


def rand_data(rng, n, dt):
    if dt == gc.F32:
        x = (rng.standard_normal(n) * rng.choice([1e-3, 1.0, 1e3])).astype(np.float32)
        x[rng.random(n) < 0.2] = 0.0
        return x
    x = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    x[rng.random(n) < rng.random()] = rng.integers(0, 8)  # runs of small values
    return x.view(NP[dt])


@pytest.mark.parametrize("case", range(CASES))
def test_fuzz(orc, case):
    rng = np.random.default_rng(1000 + case)
    op = ["scan", "iscan", "select", "partition", "pred", "split", "sort"][case % 7]
    dt = [gc.I32, gc.U32, gc.F32][int(rng.integers(0, 3))]
    off = int(rng.integers(0, 4)) if rng.random() < 0.3 else 0
    if op in ("scan", "iscan"):
        n = rand_size(rng, gc.OP_EXCLUSIVE_SCAN)
        x = (rng.integers(0, 1 << 24, size=n) * 2.0 ** -24).astype(np.float32) if dt == gc.F32 \
            else rand_data(rng, n, dt)
        xd = dev(x, off)
        f = gc.exclusive_scan if op == "scan" else gc.inclusive_scan
        want, _ = (orc.exclusive_scan if op == "scan" else orc.inclusive_scan)(x)
        out, _ = f(xd, out=empty_like_offset(xd, (off + 1) % 4))
        if dt == gc.F32:
            assert f32_within(host(out), want)[0].size == 0, (n, off)
        else:
            assert np.array_equal(host(out), want), (n, off)
    elif op in ("select", "partition"):
        n = rand_size(rng, gc.OP_SELECT_IF)
        x = rand_data(rng, n, dt)
        pred = "nonzero" if dt == gc.F32 else ["nonzero", "odd", "even"][int(rng.integers(0, 3))]
        code = {"nonzero": O.NONZERO, "odd": O.ODD, "even": O.EVEN}[pred]
        xd = dev(x, off)
        if op == "select":
            want = orc.select_if(x, code)
            out, cnt = gc.select_if(xd, pred, out=empty_like_offset(xd, (off + 3) % 4, fill=-7))
            m = int(host(cnt)[0])
            assert m == want.shape[0] and np.array_equal(host(out)[:m].view(np.uint32), want.view(np.uint32))
        else:
            want, t = orc.partition(x, code)
            out, ct = gc.partition(xd, pred, out=empty_like_offset(xd, off))
            assert int(host(ct)[0]) == t
            assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32))
    elif op == "pred":
        n = rand_size(rng, gc.OP_SELECT_IF)
        x = rand_data(rng, n, dt)
        cmp = int(rng.integers(0, 8))
        if cmp >= gc.MASK_EQ:
            mask = int(rng.integers(1, 2 ** 32))
            v = int(rng.integers(0, 2 ** 32)) & mask
        else:
            mask = 0
            v = x[int(rng.integers(0, n))].item() if rng.random() < 0.7 else \
                (float(rng.standard_normal()) if dt == gc.F32 else int(rng.integers(-2 ** 31, 2 ** 31 - 1)))
            if dt == gc.U32:
                v = int(v) % (2 ** 32)
        xd = dev(x, off)
        p = gc.predicate(xd, cmp, v, mask)
        if rng.random() < 0.5:
            want = orc.select_if_cmp(x, cmp, v, mask)
            out, cnt = gc.select_if_pred(xd, p)
            m = int(host(cnt)[0])
            assert m == want.shape[0] and np.array_equal(host(out)[:m].view(np.uint32), want.view(np.uint32))
        else:
            want, t = orc.partition_cmp(x, cmp, v, mask)
            out, ct = gc.partition_pred(xd, p)
            assert int(host(ct)[0]) == t
            assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32))
    elif op == "split":
        n = rand_size(rng, gc.OP_SPLIT_RADIX)
        keys = rand_data(rng, n, gc.U32).view(np.uint32)
        lo = int(rng.integers(0, 32))
        hi = int(rng.integers(lo, 33))
        vals = np.arange(n, dtype=np.uint32) if rng.random() < 0.5 else None
        ko, vo = gc.split_radix(dev(keys, off), dev(vals, off) if vals is not None else None, lo, hi)
        wk, wv = orc.split_radix(keys, vals, lo, hi)
        assert np.array_equal(host(ko), wk), (n, lo, hi)
        if vals is not None:
            assert np.array_equal(host(vo), wv)
    else:
        n = rand_size(rng, gc.OP_RADIX_SORT)
        keys = rand_data(rng, n, dt)
        vals = np.arange(n, dtype=np.uint32) if rng.random() < 0.7 else None
        ko, vo = gc.radix_sort(dev(keys, off), dev(vals, off) if vals is not None else None)
        wk, wv = orc.radix_sort(keys, vals)
        assert np.array_equal(host(ko).view(np.uint32), wk.view(np.uint32)), (n, dt)
        if vals is not None:
            assert np.array_equal(host(vo), wv)
