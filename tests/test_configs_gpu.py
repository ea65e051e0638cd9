"""Parity at the five benchmark configurations' full sizes, through the C ABI,
in the launch configuration bench.py times (16-byte aligned device tensors,
the persistent pipelined kernels).  Every output element is compared with
the CPU oracle: bit-exact for integer work, within 1e-5 relative (exact where
the prefix is 0) for the float32 scan against the float64 oracle.

Sizes: 2^20 - 611 (remove zeros), 10,000,000 (scans), 2^23 - 611 and the
printed 8,388,597 (keep odd), 2^28 (partition and the 1/50/99 % sweep, and
the scans at the roofline size), 2^26 (32-bit radix sort).
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import f32_within, host
from partition_pass_tile_gb300 import gc, synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def to_dev(a):
    t = torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()
    return t.view(torch.uint32) if a.dtype == np.uint32 else t


def check_select(orc, x, pred, atomic=True):
    want = orc.select_if(x, pred)
    xd = to_dev(x)
    out, cnt = gc.select_if(xd, pred)
    m = int(host(cnt)[0])
    assert m == want.shape[0]
    assert np.array_equal(host(out)[:m].view(np.uint32), want.view(np.uint32))
    if atomic:
        # one atomic per survivor (the page's comparator), then one per tile
        misplaced = []
        for per_tile in (False, True):
            out, cnt = gc.select_if_atomic(xd, pred, per_tile=per_tile)
            m2 = int(host(cnt)[0])
            got = host(out)[:m2].view(np.uint32)
            assert m2 == m
            # the comparator decides its own order: same multiset, order reported only
            assert np.array_equal(np.sort(got), np.sort(want.view(np.uint32)))
            misplaced.append(orc.count_out_of_order(got, want.view(np.uint32)))
        return misplaced
    return None


# ---------------------------------------------------------------- configuration 1

@pytest.mark.parametrize("n", [synth.SIZES["remove_zeros"], 1_049_187])
def test_config1_remove_zeros(orc, n):
    x = synth.remove_zeros(n, synth.SEEDS["remove_zeros"])
    frac = float((x == 0).mean())
    assert 0.23 < frac < 0.27  # uniform over {0,1,2,3}: about a quarter zeros
    check_select(orc, x, O.NONZERO)


# ---------------------------------------------------------------- configuration 2

def test_config2_scan_mod8_int32(orc):
    n = synth.SIZES["scan"]
    x = synth.scan_mod8(n)
    out, tot = gc.exclusive_scan(to_dev(x))
    want, wt = orc.exclusive_scan(x)
    assert np.array_equal(host(out), want)
    assert int(host(tot)[0]) == int(wt) == 45_000_000


def test_config2_scan_unit_float32(orc):
    n = synth.SIZES["scan"]
    x = synth.scan_unit_f32(n, synth.SEEDS["scan_f32"])
    out, tot = gc.exclusive_scan(to_dev(x))
    want, wt = orc.exclusive_scan(x)
    bad, worst = f32_within(host(out), want, 1e-5)
    assert bad.size == 0, (bad[:5], worst)
    assert abs(float(host(tot)[0]) - wt) <= 1e-5 * wt


def test_config2_every_fourth_two_float32_is_exact(orc):
    x = synth.every_fourth_two_f32(synth.SIZES["scan"])
    out, tot = gc.exclusive_scan(to_dev(x))
    want, wt = orc.exclusive_scan(x)
    assert np.array_equal(host(out).astype(np.float64), want)
    assert float(host(tot)[0]) == wt == 12_500_000


# ---------------------------------------------------------------- configuration 3

@pytest.mark.parametrize("n", [synth.SIZES["keep_odd"], synth.SIZES["keep_odd_literal"]])
def test_config3_keep_odd_and_atomic(orc, n):
    x = synth.uniform_i32(n, synth.SEEDS["keep_odd"])
    frac = float((x & 1).mean())
    assert 0.49 < frac < 0.51
    check_select(orc, x, O.ODD, atomic=True)


# ---------------------------------------------------------------- configuration 4

@pytest.fixture(scope="module")
def big_uniform():
    return synth.uniform_i32(synth.SIZES["partition"], synth.SEEDS["partition"])


def test_config4_partition_even(orc, big_uniform):
    x = big_uniform
    want, t = orc.partition(x, O.EVEN)
    out, ct = gc.partition(to_dev(x), "even")
    assert int(host(ct)[0]) == t
    assert np.array_equal(host(out), want)


@pytest.mark.parametrize("p,seed", [(0.01, 41), (0.50, 42), (0.99, 43)])
def test_config4_select_sweep(orc, p, seed):
    n = synth.SIZES["partition"]
    x = synth.keep_fraction(n, p, seed)
    kept = float((x != 0).mean())
    assert abs(kept - p) < 0.001
    check_select(orc, x, O.NONZERO, atomic=False)
    # both atomic comparators over the sweep: count and multiset (sorted on
    # the device, a library sort used only to compare)
    want = orc.select_if(x, O.NONZERO)
    want_sorted = torch.sort(to_dev(want.view(np.uint32)).view(torch.int32))[0]
    xd = to_dev(x)
    for per_tile in (False, True):
        out, cnt = gc.select_if_atomic(xd, "nonzero", per_tile=per_tile)
        m = int(host(cnt)[0])
        assert m == want.shape[0]
        got_sorted = torch.sort(out[:m])[0]
        assert torch.equal(got_sorted, want_sorted)


def test_config4_scans_at_roofline_size(orc, big_uniform):
    x = big_uniform
    out, tot = gc.exclusive_scan(to_dev(x))
    want, wt = orc.exclusive_scan(x)
    assert np.array_equal(host(out), want) and host(tot)[0] == wt
    del out, want
    xf = synth.scan_unit_f32(synth.SIZES["partition"], synth.SEEDS["scan_f32"])
    out, tot = gc.exclusive_scan(to_dev(xf))
    want, wt = orc.exclusive_scan(xf)
    bad, worst = f32_within(host(out), want, 1e-5)
    assert bad.size == 0, (bad[:5], worst)


# ---------------------------------------------------------------- configuration 5

def test_config5_radix_sort(orc):
    n = synth.SIZES["radix"]
    keys, vals = synth.radix_keys(n, synth.SEEDS["radix"])
    ko, vo = gc.split_radix(to_dev(keys), to_dev(vals))
    wk, wv = orc.split_radix(keys, vals)
    assert np.array_equal(host(ko), wk)
    assert np.array_equal(host(vo), wv)
    # sorted, and the payload is the permutation that sorts the input
    assert np.all(wk[1:] >= wk[:-1])
    assert np.array_equal(keys[wv], wk)
