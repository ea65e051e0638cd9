"""The largest n the C ABI accepts (GC_MAX_ELEMENTS = 2^31 - 1 elements,
8 GiB per array), checked on the device by properties that hold at any size:
the indices, tile counts and run offsets of every kernel stay in 32 bits
there.  Inputs come from a seeded torch generator on the device.
"""

import pytest
import torch

from partition_pass_tile_gb300 import gc

pytestmark = pytest.mark.gpu

N_MAX = 2 ** 31 - 1


def seeded_small_ints(n, seed, high):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(0, high, (n,), dtype=torch.int32, device="cuda", generator=g)


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_scan_at_max_n():
    x = seeded_small_ints(N_MAX, 71, 8)
    ws = gc.workspace(gc.OP_EXCLUSIVE_SCAN, N_MAX)
    out, total = gc.exclusive_scan(x, ws=ws)
    assert int(out[0]) == 0
    # out[i + 1] - out[i] == x[i] modulo 2^32 (int32 arithmetic wraps)
    assert bool(torch.equal(out[1:] - out[:-1], x[:-1]))
    assert int(total[0]) == int((out[-1] + x[-1]).item())
    # the true sum, reduced to int32 the way the scan wraps
    s64 = int(x.to(torch.int64).sum())
    assert int(total[0]) == (s64 + 2 ** 31) % 2 ** 32 - 2 ** 31
    assert gc.query_device_status(ws) == 0


def test_select_and_partition_at_max_n():
    x = seeded_small_ints(N_MAX, 72, 8)
    out, count = gc.select_if(x, "nonzero")
    keep = x != 0
    m = int(keep.sum())
    assert int(count[0]) == m
    assert bool(torch.equal(out[:m], x[keep]))
    del out, keep
    torch.cuda.empty_cache()
    out, count_true = gc.partition(x, "even")
    even = (x & 1) == 0
    t = int(even.sum())
    assert int(count_true[0]) == t
    assert bool(torch.equal(out[:t], x[even]))
    assert bool(torch.equal(out[t:], x[~even]))


@pytest.mark.parametrize("sort", ["split_radix", "radix_sort"])
def test_radix_at_max_n(sort):
    g = torch.Generator(device="cuda")
    g.manual_seed(73)
    keys = torch.randint(0, 2 ** 31 - 1, (N_MAX,), dtype=torch.int32, device="cuda", generator=g)
    vals = torch.arange(N_MAX, dtype=torch.int32, device="cuda")
    if sort == "split_radix":
        ko, vo = gc.split_radix(keys.view(torch.uint32), vals.view(torch.uint32), 0, 32)
    else:
        ko, vo = gc.radix_sort(keys, vals.view(torch.uint32))
    del vals
    torch.cuda.empty_cache()
    ko, vo = ko.view(torch.int32), vo.view(torch.int32)
    assert bool((ko[1:] >= ko[:-1]).all())  # keys below 2^31: signed order = unsigned order
    # stable: equal keys keep their payloads (original indices) ascending
    assert not bool(((ko[1:] == ko[:-1]) & (vo[1:] <= vo[:-1])).any())
    # each output key is the input key at its payload's index ...
    assert bool(torch.equal(torch.index_select(keys, 0, vo), ko))
    # ... and the payloads are a permutation of 0 .. n-1: sum and sum of
    # squares against their closed forms, both modulo 2^64 (int64 sums wrap)
    v64 = vo.to(torch.int64)
    n = N_MAX

    def wrap64(v):
        return (v + 2 ** 63) % 2 ** 64 - 2 ** 63

    assert int(v64.sum()) == n * (n - 1) // 2
    assert int((v64 * v64).sum()) == wrap64((n - 1) * n * (2 * n - 1) // 6)
