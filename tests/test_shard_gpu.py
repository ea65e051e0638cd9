"""The sharded path on one GPU: P shards of one array computed one after
another through gc_reduce / gc_count_if, gc_shard_offsets and the placed
passes (gc_exclusive_scan_carry, gc_select_if_at, gc_partition_at), the
concatenated result compared with the oracle on the whole array.

On one GPU the exchange is the P pre-pass results written into the P slots of
one device array; across GPUs it is the all-gather of partition_pass_tile_
gb300.shard.gather_totals.  Shards start at arbitrary element offsets, so most
of them are 4-byte but not 16-byte aligned and run the persistent kernels'
shifted instantiations (staged from the 16-byte boundary below the shard),
the others the aligned ones.  Bit-exact for integers, 1e-5 relative (exact at
a zero prefix) for float32 against the float64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import dev, f32_within, host
from partition_pass_tile_gb300 import gc, shard, synth

pytestmark = pytest.mark.gpu

SIZES = [1, 1000, 100_003, 3 * 8192 + 611, 1_047_965]
PARTS = [1, 2, 3, 7]


def _input(n, dt, seed):
    if dt == gc.F32:
        return synth.scan_unit_f32(n, seed)
    x = synth.uniform_u32(n, seed) if dt == gc.U32 else synth.uniform_i32(n, seed)
    return x


@pytest.mark.parametrize("parts", PARTS)
@pytest.mark.parametrize("dt", [gc.I32, gc.U32, gc.F32])
def test_sharded_exclusive_scan(orc, parts, dt):
    for n in SIZES:
        x = _input(n, dt, 31 + n % 7)
        xd = dev(x)
        out = torch.empty_like(xd)
        totals = torch.empty(parts, dtype=xd.dtype, device="cuda")
        ends = torch.empty(parts, dtype=xd.dtype, device="cuda")
        bounds = [shard.shard_bounds(n, parts, r) for r in range(parts)]
        for r, (a, b) in enumerate(bounds):          # pre-pass of every shard
            gc.reduce(xd[a:b], total=totals[r:r + 1])
        for r, (a, b) in enumerate(bounds):          # offsets, then the placed scan
            carry = gc.shard_offsets(gc.OP_EXCLUSIVE_SCAN, totals, r)
            gc.exclusive_scan_carry(xd[a:b], carry, out=out[a:b], total=ends[r:r + 1])
        want, wtot = orc.exclusive_scan(x)
        got = host(out)
        last = host(ends)[-1]
        if dt == gc.F32:
            bad, worst = f32_within(got, want)
            assert bad.size == 0, (n, parts, bad[:5], worst)
            assert abs(float(last) - wtot) <= 1e-5 * abs(wtot)
        else:
            assert np.array_equal(got, want), (n, parts)
            assert last == wtot
        # every shard's total is its own reduction, and shard r's end is the
        # carry of shard r + 1
        if dt != gc.F32:
            for r, (a, b) in enumerate(bounds):
                assert host(totals)[r] == orc.exclusive_scan(x[a:b])[1]


@pytest.mark.parametrize("parts", PARTS)
@pytest.mark.parametrize("dt,pred", [(gc.I32, gc.NONZERO), (gc.U32, gc.ODD), (gc.F32, gc.NONZERO)])
def test_sharded_select_if(orc, parts, dt, pred):
    for n in SIZES:
        x = synth.keep_fraction(n, 0.37, 41 + n % 5)
        if dt == gc.F32:
            x = np.where(x != 0, synth.scan_unit_f32(n, 3) + np.float32(0.5), np.float32(0.0)).astype(np.float32)
        elif dt == gc.U32:
            x = x.view(np.uint32)
        xd = dev(x)
        base = torch.full((n + 8,), -1, dtype=torch.int32, device="cuda")
        out = base[:n].view(xd.dtype) if dt != gc.I32 else base[:n]
        counts = torch.empty(parts, dtype=torch.uint32, device="cuda")
        own = torch.empty(parts, dtype=torch.uint32, device="cuda")
        bounds = [shard.shard_bounds(n, parts, r) for r in range(parts)]
        for r, (a, b) in enumerate(bounds):
            gc.count_if(xd[a:b], pred, count=counts[r:r + 1])
        for r, (a, b) in enumerate(bounds):
            off = gc.shard_offsets(gc.OP_SELECT_IF, counts, r, dtype=gc.U32)
            gc.select_if_at(xd[a:b], pred, out, off, count=own[r:r + 1])
        want = orc.select_if(x, pred)
        m = want.shape[0]
        assert int(host(counts).astype(np.int64).sum()) == m
        assert np.array_equal(host(own), host(counts))
        got = host(base)
        assert np.array_equal(got[:m].view(np.uint32), want.view(np.uint32)), (n, parts)
        assert np.all(got[m:] == -1)  # nothing past the survivors, nor past out


@pytest.mark.parametrize("parts", PARTS)
@pytest.mark.parametrize("dt,pred", [(gc.I32, gc.EVEN), (gc.U32, gc.ODD), (gc.F32, gc.NONZERO)])
def test_sharded_partition(orc, parts, dt, pred):
    for n in SIZES:
        if dt == gc.F32:
            x = synth.scan_unit_f32(n, 5)
            x[synth.uniform_u32(n, 6) % 3 == 0] = 0.0
        else:
            x = _input(n, dt, 51 + n % 3)
        xd = dev(x)
        out = torch.empty_like(xd)
        counts = torch.empty(parts, dtype=torch.uint32, device="cuda")
        own = torch.empty(parts, dtype=torch.uint32, device="cuda")
        bounds = [shard.shard_bounds(n, parts, r) for r in range(parts)]
        sizes = [b - a for a, b in bounds]
        for r, (a, b) in enumerate(bounds):
            gc.count_if(xd[a:b], pred, count=counts[r:r + 1])
        for r, (a, b) in enumerate(bounds):
            offs = gc.shard_offsets(gc.OP_PARTITION, counts, r, sizes=sizes, dtype=gc.U32)
            gc.partition_at(xd[a:b], pred, out, offs, count_true=own[r:r + 1])
        want, t = orc.partition(x, pred)
        assert int(host(counts).astype(np.int64).sum()) == t
        assert np.array_equal(host(own), host(counts))
        assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32)), (n, parts)


def test_shard_offsets_values():
    """The offsets kernel on hand-made totals: exclusive sums, the partition's
    rejected start T + sizes before - kept before, and a wrapping int sum."""
    counts = torch.tensor([5, 0, 7, 2], dtype=torch.int32, device="cuda").view(torch.uint32)
    sizes = [10, 3, 9, 4]
    for r, want in enumerate([0, 5, 5, 12]):
        assert int(gc.shard_offsets(gc.OP_SELECT_IF, counts, r, dtype=gc.U32).item()) == want
    T = 14
    for r in range(4):
        kb = sum([5, 0, 7, 2][:r])
        got = gc.shard_offsets(gc.OP_PARTITION, counts, r, sizes=sizes, dtype=gc.U32).cpu().tolist()
        assert got == [kb, T + sum(sizes[:r]) - kb]
    big = torch.tensor([0x7FFFFFFF, 0x7FFFFFFF, 5], dtype=torch.int32, device="cuda")
    assert int(gc.shard_offsets(gc.OP_EXCLUSIVE_SCAN, big, 2).item()) == -2  # modulo 2^32
    f = torch.tensor([0.5, 0.25, 1.0], dtype=torch.float32, device="cuda")
    assert float(gc.shard_offsets(gc.OP_EXCLUSIVE_SCAN, f, 2).item()) == 0.75


def test_placed_run_past_capacity_is_refused():
    """A base that puts the survivors past out's capacity: the kernel writes
    nothing there and the status query reports GC_ERR_DEVICE_CHECK."""
    n = 100_003
    x = synth.keep_fraction(n, 0.5, 9)
    xd = dev(x)
    big = torch.full((n + 64,), -1, dtype=torch.int32, device="cuda")
    cap = 1000
    base = torch.tensor([cap - 10], dtype=torch.int64, device="cuda")
    ws = gc.workspace(gc.OP_SELECT_IF, n)
    gc.select_if_at(xd, gc.NONZERO, big[:cap], base, ws=ws)
    assert gc.query_device_status(ws) == 7  # GC_ERR_DEVICE_CHECK
    assert np.all(host(big)[cap:] == -1)
    # the workspace serves a correct call afterwards
    base.zero_()
    out, cnt = gc.select_if_at(xd, gc.NONZERO, big[:n], base, ws=ws)
    assert gc.query_device_status(ws) == 0
    want = x[x != 0]
    assert int(host(cnt)[0]) == want.size
    assert np.array_equal(host(big)[:want.size], want)
