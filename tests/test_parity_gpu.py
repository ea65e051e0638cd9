"""Parity of every libgc entry point with the CPU oracle, on the GPU, through the C ABI.

Integer results must be bit-exact; float32 scans must be within 1e-5 relative
of the float64 oracle (exact where the oracle prefix is 0).  Sizes span one
element, warp and vector boundaries, exact tiles and ragged tails; 16-byte
aligned tensors take the vector kernels and offset tensors the scalar ones.
"""

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import dev, empty_like_offset, f32_within, host
from partition_pass_tile_gb300 import gc, synth

pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(2024)
NP = {gc.I32: np.int32, gc.U32: np.uint32, gc.F32: np.float32}


def sizes_for(op):
    T = gc.tile_elements(op)
    return sorted({1, 2, 3, 4, 5, 31, 32, 33, 127, 128, 129, 1023, 1024, 1025, T - 1, T, T + 1,
                   2 * T - 1, 2 * T + 3, 33 * T + 17, 100_003})


def rand(n, dt, kind="wide"):
    if dt == gc.F32:
        return synth.scan_unit_f32(n, int(RNG.integers(1 << 30)))
    if kind == "small":
        return RNG.integers(-3, 4, size=n).astype(NP[dt]) if dt == gc.I32 else \
            RNG.integers(0, 4, size=n).astype(np.uint32)
    return synth.uniform_u32(n, int(RNG.integers(1 << 30))).view(NP[dt])


# ---------------------------------------------------------------- scan

@pytest.mark.parametrize("dt", [gc.I32, gc.U32, gc.F32])
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_scan_sizes(orc, dt, offset):
    for n in sizes_for(gc.OP_EXCLUSIVE_SCAN):
        x = rand(n, dt)
        want, want_total = orc.exclusive_scan(x)
        xd = dev(x, offset)
        out = empty_like_offset(xd, offset)
        out, tot = gc.exclusive_scan(xd, out=out)
        got = host(out)
        if dt == gc.F32:
            bad, worst = f32_within(got, want)
            assert bad.size == 0, (n, bad[:5], worst)
            tb, _ = f32_within(host(tot), np.array([want_total]))
            assert tb.size == 0
        else:
            assert np.array_equal(got, want), (n, np.flatnonzero(got != want)[:5])
            assert host(tot)[0] == want_total


@pytest.mark.parametrize("dt", [gc.I32, gc.F32])
def test_scan_in_place(orc, dt):
    n = 3 * gc.tile_elements(gc.OP_EXCLUSIVE_SCAN) + 5
    x = rand(n, dt)
    want, _ = orc.exclusive_scan(x)
    xd = dev(x)
    gc.exclusive_scan(xd, out=xd)
    got = host(xd)
    if dt == gc.F32:
        assert f32_within(got, want)[0].size == 0
    else:
        assert np.array_equal(got, want)


def test_scan_wraps_and_empty(orc):
    x = np.full(50_000, 0xFFFFFFF0, dtype=np.uint32)
    want, wt = orc.exclusive_scan(x)
    out, tot = gc.exclusive_scan(dev(x))
    assert np.array_equal(host(out), want) and host(tot)[0] == wt
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    tot = torch.full((1,), 77, dtype=torch.int32, device="cuda")
    gc.exclusive_scan(e, out=e.clone(), total=tot)
    assert tot.item() == 0


def test_scan_f32_exact_inputs_are_exact(orc):
    """Every-fourth-is-2 (Day 32): all prefixes are integers < 2^24, so the
    float32 scan must be exact whatever the summation order."""
    x = synth.every_fourth_two_f32(1_000_000)
    want, _ = orc.exclusive_scan(x)
    out, tot = gc.exclusive_scan(dev(x))
    assert np.array_equal(host(out).astype(np.float64), want)
    assert host(tot)[0] == 1_250_000


# ---------------------------------------------------------------- select-if

CASES = [(gc.I32, gc.NONZERO), (gc.I32, gc.ODD), (gc.I32, gc.EVEN), (gc.U32, gc.NONZERO),
         (gc.U32, gc.ODD), (gc.U32, gc.EVEN), (gc.F32, gc.NONZERO)]


def select_input(n, dt):
    if dt == gc.F32:
        x = synth.scan_unit_f32(n, int(RNG.integers(1 << 30)))
        x[RNG.random(n) < 0.3] = 0.0
        x[RNG.random(n) < 0.05] = -0.0
        return x
    return rand(n, dt, "small")


@pytest.mark.parametrize("dt,pred", CASES)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_select_sizes(orc, dt, pred, offset):
    for n in sizes_for(gc.OP_SELECT_IF):
        x = select_input(n, dt)
        want = orc.select_if(x, pred)
        xd = dev(x, offset)
        out = empty_like_offset(xd, (offset + 1) % 4, fill=-7)
        sentinel = host(out[:1]).view(np.uint32)[0]
        out, cnt = gc.select_if(xd, pred, out=out)
        m = int(host(cnt)[0])
        got = host(out).view(np.uint32)
        assert m == want.shape[0], (n, m, want.shape[0])
        assert np.array_equal(got[:m], want.view(np.uint32)), n
        assert np.all(got[m:] == sentinel), "wrote past the survivors"


def test_select_all_and_none():
    T = gc.tile_elements(gc.OP_SELECT_IF)
    for n in (1, T, 5 * T + 9):
        ones = np.arange(1, n + 1, dtype=np.int32)
        out, cnt = gc.select_if(dev(ones), "nonzero")
        assert host(cnt)[0] == n and np.array_equal(host(out), ones)
        out, cnt = gc.select_if(dev(np.zeros(n, np.int32)), "nonzero")
        assert host(cnt)[0] == 0


def test_select_float_special_values(orc):
    x = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1e-45, -1e-45, 2.5] * 1000, dtype=np.float32)
    want = orc.select_if(x, O.NONZERO)
    out, cnt = gc.select_if(dev(x), "nonzero")
    m = int(host(cnt)[0])
    assert m == want.shape[0] == 6000
    assert np.array_equal(host(out)[:m].view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------- partition

@pytest.mark.parametrize("dt,pred", CASES)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_partition_sizes(orc, dt, pred, offset):
    for n in sizes_for(gc.OP_PARTITION):
        x = select_input(n, dt) if dt == gc.F32 else rand(n, dt, "wide")
        want, t = orc.partition(x, pred)
        xd = dev(x, offset)
        out = empty_like_offset(xd, (offset + 3) % 4)
        out, ct = gc.partition(xd, pred, out=out)
        assert int(host(ct)[0]) == t, n
        assert np.array_equal(host(out).view(np.uint32), want.view(np.uint32)), n


# ---------------------------------------------------------------- radix

@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_radix_full_sort(orc, offset):
    for n in [1, 2, 33, 4095, 4097, 100_003, 300_001]:
        keys = synth.uniform_u32(n, int(RNG.integers(1 << 30)))
        keys[::5] = keys[0]
        vals = np.arange(n, dtype=np.uint32)
        wk, wv = orc.split_radix(keys, vals)
        kd, vd = dev(keys, offset), dev(vals, offset)
        ko, vo = gc.split_radix(kd, vd, keys_out=empty_like_offset(kd, offset),
                                vals_out=empty_like_offset(vd, offset))
        assert np.array_equal(host(ko), wk) and np.array_equal(host(vo), wv), n


def test_radix_bit_ranges_keys_only_and_in_place(orc):
    n = 70_001
    keys = synth.uniform_u32(n, 99)
    vals = np.arange(n, dtype=np.uint32)
    for b, e in [(0, 1), (7, 8), (31, 32), (4, 12), (0, 7), (3, 3)]:
        wk, wv = orc.split_radix(keys, vals, b, e)
        ko, vo = gc.split_radix(dev(keys), dev(vals), b, e)
        assert np.array_equal(host(ko), wk) and np.array_equal(host(vo), wv), (b, e)
        ko, _ = gc.split_radix(dev(keys), None, b, e)
        assert np.array_equal(host(ko), wk), (b, e)
    for b, e in [(0, 32), (0, 31), (5, 6)]:          # in place, even and odd bit counts
        wk, wv = orc.split_radix(keys, vals, b, e)
        kd, vd = dev(keys), dev(vals)
        gc.split_radix(kd, vd, b, e, keys_out=kd, vals_out=vd)
        assert np.array_equal(host(kd), wk) and np.array_equal(host(vd), wv), (b, e)


def test_radix_degenerate(orc):
    n = 10_000
    eq = np.full(n, 7, dtype=np.uint32)
    idx = np.arange(n, dtype=np.uint32)
    ko, vo = gc.split_radix(dev(eq), dev(idx))
    assert np.array_equal(host(ko), eq) and np.array_equal(host(vo), idx)
    srt = np.sort(synth.uniform_u32(n, 3))
    ko, vo = gc.split_radix(dev(srt), dev(idx))
    assert np.array_equal(host(ko), srt) and np.array_equal(host(vo), idx)


# ---------------------------------------------------------------- atomic comparator

@pytest.mark.parametrize("per_tile", [False, True], ids=["per_survivor", "per_tile"])
@pytest.mark.parametrize("dt,pred", CASES)
def test_atomic_multiset(orc, dt, pred, per_tile):
    # several correct answers: the count and the multiset are unique, the order is not
    for n in [1, 3, 33, 4097, 100_003]:
        for off in (0, 1):
            x = select_input(n, dt)
            want = orc.select_if(x, pred)
            out = empty_like_offset(dev(x), off, fill=-1)
            cnt = torch.full((1,), 12345, dtype=torch.int32, device="cuda").view(torch.uint32)
            gc.select_if_atomic(dev(x, off), pred, out=out, count=cnt, per_tile=per_tile)
            m = int(host(cnt)[0])
            got = host(out)
            assert m == want.shape[0]
            assert np.array_equal(np.sort(got[:m].view(np.uint32)), np.sort(want.view(np.uint32)))
            sentinel = host(empty_like_offset(dev(x[:1]), 0, fill=-1))[0]
            assert np.all(got[m:] == sentinel)  # nothing written past the survivors


# ---------------------------------------------------------------- workspace reuse

def test_one_workspace_serves_every_op(orc):
    n = 200_001
    ws = gc.workspace(gc.OP_SPLIT_RADIX, n)
    assert ws.numel() >= max(gc.workspace_bytes(op, n, gc.F32) for op in range(5))
    x = synth.uniform_i32(n, 8)
    xf = synth.scan_unit_f32(n, 8)
    for _ in range(2):
        out, _ = gc.exclusive_scan(dev(x), ws=ws)
        assert np.array_equal(host(out), orc.exclusive_scan(x)[0])
        out, _ = gc.exclusive_scan(dev(xf), ws=ws)
        assert f32_within(host(out), orc.exclusive_scan(xf)[0])[0].size == 0
        out, c = gc.select_if(dev(x), "odd", ws=ws)
        w = orc.select_if(x, O.ODD)
        assert np.array_equal(host(out)[: int(host(c)[0])], w)
        out, c = gc.partition(dev(x), "even", ws=ws)
        assert np.array_equal(host(out), orc.partition(x, O.EVEN)[0])
        ko, _ = gc.split_radix(dev(x.view(np.uint32)), None, ws=ws)
        assert np.array_equal(host(ko), orc.split_radix(x.view(np.uint32))[0])
        assert gc.query_device_status(ws) == 0


def test_workspace_reuse_small_sort_then_large_scan(orc):
    """A workspace sized for the largest call, first used by small radix sorts
    (whose ping-pong buffers and digit table sit where a much larger call's
    status words go), then by a 64x larger scan and select: every call clears
    its own status words, whatever the workspace held before."""
    small, big = 100_003, 64 * 100_003
    ws = gc.workspace(gc.OP_RADIX_SORT, big, gc.F32)
    assert ws.numel() >= max(gc.workspace_bytes(op, big, gc.F32) for op in range(7))
    keys, vals = synth.radix_keys(small, 9)
    ko, vo = gc.split_radix(dev(keys), dev(vals), ws=ws)
    assert np.array_equal(host(ko), orc.split_radix(keys, vals)[0])
    kf = synth.scan_unit_f32(small, 9) - np.float32(0.5)
    ko, _ = gc.radix_sort(dev(kf), None, ws=ws)
    assert np.array_equal(host(ko).view(np.uint32), orc.radix_sort(kf)[0].view(np.uint32))
    xf = synth.scan_unit_f32(big, 10)
    out, _ = gc.exclusive_scan(dev(xf), ws=ws)
    assert f32_within(host(out), orc.exclusive_scan(xf)[0])[0].size == 0
    x = synth.uniform_i32(big, 10)
    out, c = gc.select_if(dev(x), "odd", ws=ws)
    w = orc.select_if(x, O.ODD)
    assert int(host(c)[0]) == w.shape[0] and np.array_equal(host(out)[: w.shape[0]], w)
    assert gc.query_device_status(ws) == 0


def test_back_to_back_calls_alternating_inputs(orc):
    """Persistent calls clear their status words inside the kernel, behind a
    start barrier.  Back-to-back calls on one workspace with inputs that
    alternate (so that a status word left by the previous call would give a
    different prefix), all results kept on the device and checked at the end:
    a tile that read a word before its clear would show as a wrong prefix."""
    n = 5_000_011  # more tiles than the persistent grid has CTAs
    xs = [synth.uniform_i32(n, 31), synth.scan_mod8(n)]
    ks = [synth.keep_fraction(n, 0.25, 32), synth.keep_fraction(n, 0.75, 33)]
    xd, kd = [dev(a) for a in xs], [dev(a) for a in ks]
    ws = gc.workspace(gc.OP_SELECT_IF, n)
    scans, sels = [], []
    for i in range(12):
        scans.append(gc.exclusive_scan(xd[i % 2], ws=ws)[0])
        sels.append(gc.select_if(kd[i % 2], "nonzero", ws=ws))
    want_scan = [orc.exclusive_scan(a)[0] for a in xs]
    want_sel = [orc.select_if(a, O.NONZERO) for a in ks]
    for i in range(12):
        assert np.array_equal(host(scans[i]), want_scan[i % 2]), i
        out, c = sels[i]
        w = want_sel[i % 2]
        assert int(host(c)[0]) == w.shape[0] and np.array_equal(host(out)[: w.shape[0]], w), i
    assert gc.query_device_status(ws) == 0


def test_streams_and_empty_inputs():
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        x = torch.arange(1, 10_001, dtype=torch.int32, device="cuda")
        out, tot = gc.exclusive_scan(x, stream=s)
    s.synchronize()
    assert tot.item() == 10_000 * 10_001 // 2
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    c = torch.full((1,), 5, dtype=torch.int32, device="cuda").view(torch.uint32)
    gc.select_if(e, "odd", out=e.clone(), count=c)
    assert c.view(torch.int32).item() == 0
    c.view(torch.int32).fill_(5)
    gc.partition(e, "odd", out=e.clone(), count_true=c)
    assert c.view(torch.int32).item() == 0


# ---------------------------------------------------------------- one tile per CTA

def test_fallback_kernels_match_oracle(orc):
    """The one-tile-per-CTA kernels (run when the device refuses a cooperative
    grid), forced by the test hook, on ragged sizes with aligned and offset
    pointers: scan, select-if, partition and the one-bit split."""
    gc.testing_force_fallback(True)
    try:
        for n in (1, 1000, 3 * 8192 + 611, 100_003):
            for off in (0, 1, 2):
                x = rand(n, gc.I32, "small")
                out, tot = gc.exclusive_scan(dev(x, off), out=empty_like_offset(dev(x), (off + 1) % 4))
                want, wt = orc.exclusive_scan(x)
                assert np.array_equal(host(out), want) and host(tot)[0] == wt, (n, off)
                xf = synth.scan_unit_f32(n, 3)
                out, _ = gc.exclusive_scan(dev(xf, off))
                assert f32_within(host(out), orc.exclusive_scan(xf)[0])[0].size == 0, (n, off)
                y = select_input(n, gc.I32)
                out, cnt = gc.select_if(dev(y, off), gc.ODD)
                want = orc.select_if(y, gc.ODD)
                m = int(host(cnt)[0])
                assert m == want.shape[0] and np.array_equal(host(out)[:m], want), (n, off)
                out, ct = gc.partition(dev(x, off), gc.EVEN)
                want, t = orc.partition(x, gc.EVEN)
                assert int(host(ct)[0]) == t and np.array_equal(host(out), want), (n, off)
                k = synth.uniform_u32(n, 4)
                v = np.arange(n, dtype=np.uint32)
                ko, vo = gc.split_radix(dev(k, off), dev(v, off), 0, 4)
                wk, wv = orc.split_radix(k, v, 0, 4)
                assert np.array_equal(host(ko), wk) and np.array_equal(host(vo), wv), (n, off)
    finally:
        gc.testing_force_fallback(False)
