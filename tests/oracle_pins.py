"""Pins for the CPU oracle: facts fixed by the pages or by mathematics, not by the oracle.

Every pin is a function ``pin_*(o)`` that takes an ``oracle.Oracle`` and raises
AssertionError when the oracle disagrees with the fact.  ``test_oracle_pins.py``
runs them against the real oracle (all must pass) and against deliberately
broken copies of oracle.c (each copy must fail at least one pin).

Nothing here calls the oracle to make an expected value: every expected value
is printed on a page (tests/golden/), a closed form, a brute-force count
written independently in Python, or a numpy library routine.
"""

from __future__ import annotations

import numpy as np

import oracle as O
from conftest import load_golden
from partition_pass_tile_gb300 import synth


def _py_keep(v: int, dtype: str, pred: int) -> bool:
    """Predicate restated in plain Python (independent of oracle.c)."""
    if pred == O.NONZERO:
        return v != 0  # for floats v is a Python float: -0.0 == 0, nan != 0
    if pred == O.ODD:
        return (int(v) & 1) == 1
    return (int(v) & 1) == 0


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- scan, integer

def pin_scan_printed_head(o):
    """CIS 565 scan log: the 13 printed inputs give the 13 printed outputs."""
    g = load_golden("cis565_scan_log.txt")
    x = np.array(g["input_head"], dtype=np.int32)
    out, tot = o.exclusive_scan(x)
    assert out.tolist() == g["pot_out_head"], out
    assert out.tolist() == g["npot_out_head"]
    assert int(tot) == g["pot_out_head"][-1] + g["input_head"][-1]


def pin_scan_printed_full(o):
    """CIS 565 scan log, whole arrays.  The printed tail inputs and the
    printed output tails fix in[247..255] and the sums of the elided middle;
    any middle with those sums must reproduce every printed output value for
    both the 256-element and the 253-element run."""
    g = load_golden("cis565_scan_log.txt")
    head, tail = g["input_head"], g["input_tail"]
    pot_tail, npot_tail = g["pot_out_tail"], g["npot_out_tail"]
    n = g["pot_n"][0]
    x = np.zeros(n, dtype=np.int64)
    x[: len(head)] = head
    x[n - len(tail):] = tail
    # npot_out_tail covers out[247..252]; consecutive differences are inputs
    # 247..251, the last of which overlap the printed input tail.
    d = np.diff(np.array(npot_tail, dtype=np.int64))
    x[247:247 + len(d)] = d
    assert x[250] == tail[0] and x[251] == tail[1]
    # fill in[13..246] with values in 0..49 whose sum is out[247] - out[13]
    s13 = sum(head)
    need = npot_tail[0] - s13
    k = 247 - len(head)
    base, extra = divmod(need, k)
    mid = np.full(k, base, dtype=np.int64)
    mid[:extra] += 1
    assert 0 <= mid.min() and mid.max() <= 49
    x[len(head):247] = mid
    x = x.astype(np.int32)
    out, tot = o.exclusive_scan(x)
    assert out[: len(head)].tolist() == g["pot_out_head"]
    assert out[n - len(pot_tail):].tolist() == pot_tail
    npot = g["npot_n"][0]
    out2, _ = o.exclusive_scan(x[:npot])
    assert out2[npot - len(npot_tail):].tolist() == npot_tail
    assert out2[: len(head)].tolist() == g["npot_out_head"]
    assert int(tot) == pot_tail[-1] + tail[-1]


def pin_scan_mod8_closed_form(o, n=10_000_000):
    """(i % 8) + 1: exclusive prefix 36*floor(i/8) + r(r+1)/2 with r = i % 8,
    total 4.5 n for n a multiple of 8 (45,000,000 at ten million)."""
    x = synth.scan_mod8(n)
    out, tot = o.exclusive_scan(x)
    i = np.arange(n, dtype=np.int64)
    r = i % 8
    want = 36 * (i // 8) + r * (r + 1) // 2
    assert np.array_equal(out.astype(np.int64), want)
    assert int(tot) == 45_000_000


def pin_scan_every_fourth_two(o):
    """Day 32 input: every fourth element 2, the rest 1.  Prefix is
    i + ceil(i / 4); total 12,500,000; exact in float32 and in int32."""
    g = load_golden("day32_every_fourth_two.txt")
    n = g["n"][0]
    xf = synth.every_fourth_two_f32(n)
    assert int((xf == 2.0).sum()) == g["twos"][0]
    i = np.arange(n, dtype=np.int64)
    want = i + (i + 3) // 4
    outf, totf = o.exclusive_scan(xf)
    assert totf == g["total"][0]
    assert np.array_equal(outf, want.astype(np.float64))
    outi, toti = o.exclusive_scan(xf.astype(np.int32))
    assert np.array_equal(outi.astype(np.int64), want)
    assert int(toti) == g["total"][0]


def pin_scan_wraps_mod_2_32(o):
    """Integer adds wrap modulo 2^32 (the same bits for int32 and uint32)."""
    x = np.array([0xFFFFFFFF, 2, 5, 0x80000000, 0x80000000], dtype=np.uint32)
    out, tot = o.exclusive_scan(x)
    assert out.tolist() == [0, 0xFFFFFFFF, 1, 6, 0x80000006]
    assert int(tot) == 6
    out_i, tot_i = o.exclusive_scan(x.view(np.int32))
    assert np.array_equal(out_i.view(np.uint32), out)
    assert int(tot_i) == 6


def pin_scan_brute_force(o):
    """out[i] = sum of in[0..i-1] mod 2^32, by Python big-int sums, n <= 300."""
    rng = _rng(11)
    for n in [0, 1, 2, 3, 7, 31, 32, 33, 100, 255, 256, 257, 300]:
        x = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
        out, tot = o.exclusive_scan(x)
        vals = [int(v) for v in x]
        for i in range(n):
            assert int(out[i]) == sum(vals[:i]) % 2 ** 32, (n, i)
        assert int(tot) == sum(vals) % 2 ** 32


def pin_scan_first_difference(o):
    """out[i+1] - out[i] = in[i] (mod 2^32) and out[0] = 0."""
    x = synth.uniform_u32(100_003, 7)
    out, tot = o.exclusive_scan(x)
    assert out[0] == 0
    with np.errstate(over="ignore"):
        assert np.array_equal(out[1:] - out[:-1], x[:-1])
        assert np.uint32(tot) == out[-1] + x[-1]


def pin_inclusive_is_shifted_exclusive(o):
    """inclusive[i] = exclusive[i] + in[i], both totals equal."""
    x = synth.uniform_u32(5_001, 9)
    ex, t1 = o.exclusive_scan(x)
    inc, t2 = o.inclusive_scan(x)
    with np.errstate(over="ignore"):
        assert np.array_equal(inc, ex + x)
    assert int(t1) == int(t2)
    xf = synth.scan_unit_f32(5_001, 9)
    exf, _ = o.exclusive_scan(xf)
    incf, _ = o.inclusive_scan(xf)
    assert np.array_equal(incf, exf + xf.astype(np.float64))


# ------------------------------------------------------------------ scan, float

def pin_scan_f32_exact(o, n=1_000_003):
    """Inputs k * 2^-24 with integer k: the double prefix must equal the
    integer prefix of k (numpy cumsum over int64) times 2^-24, exactly."""
    x = synth.scan_unit_f32(n, 2)
    k = (x.astype(np.float64) * 2.0 ** 24).astype(np.int64)
    assert np.array_equal(k.astype(np.float64) * 2.0 ** -24, x.astype(np.float64))
    want = np.concatenate([[0], np.cumsum(k)[:-1]]).astype(np.float64) * 2.0 ** -24
    out, tot = o.exclusive_scan(x)
    assert np.array_equal(out, want)
    assert tot == float(k.sum()) * 2.0 ** -24


def pin_scan_f32_small_closed_form(o):
    """Hand values: [0.5, 0.25, 1.0, 3.0] -> [0, 0.5, 0.75, 1.75], total 4.75."""
    out, tot = o.exclusive_scan(np.array([0.5, 0.25, 1.0, 3.0], dtype=np.float32))
    assert out.tolist() == [0.0, 0.5, 0.75, 1.75] and tot == 4.75


# ------------------------------------------------------------------ select-if

def pin_select_printed(o):
    """CIS 565 compaction log: zeros removed, order kept, head and tail."""
    g = load_golden("cis565_compact_log.txt")
    head = np.array(g["input_head"], dtype=np.int32)
    got = o.select_if(head, O.NONZERO)
    nz = int((head != 0).sum())
    assert got.tolist() == g["pot_out_head"][:nz]
    tail = np.array(g["input_tail"], dtype=np.int32)
    assert o.select_if(tail, O.NONZERO).tolist() == g["pot_out_tail"][1:]
    # the 253-element run ends at input 252, the third printed tail input
    npot_last = tail[: g["npot_n"][0] - (g["pot_n"][0] - len(tail))]
    got_npot = o.select_if(npot_last, O.NONZERO).tolist()
    assert got_npot == g["npot_out_tail"][-len(got_npot):]


def _brute_select(vals, dtype, pred):
    n = len(vals)
    keep = [_py_keep(v, dtype, pred) for v in vals]
    m = sum(keep)
    out = [None] * m
    for i in range(n):
        if keep[i]:
            rank = sum(1 for j in range(i) if keep[j])  # O(n^2) on purpose
            out[rank] = vals[i]
    return out


def pin_select_brute_force(o):
    """out[rank[i]] = in[i] with rank[i] = #{j < i : keep(in[j])}, O(n^2)."""
    rng = _rng(12)
    for n in [0, 1, 2, 5, 31, 32, 33, 64, 129, 200]:
        xi = rng.integers(-3, 4, size=n).astype(np.int32)
        for pred in (O.NONZERO, O.ODD, O.EVEN):
            want = _brute_select([int(v) for v in xi], "i32", pred)
            assert o.select_if(xi, pred).tolist() == want, (n, pred)
            assert o.count_if(xi, pred) == len(want)
        xu = xi.view(np.uint32)
        for pred in (O.NONZERO, O.ODD, O.EVEN):
            want = _brute_select([int(v) for v in xu], "u32", pred)
            assert o.select_if(xu, pred).tolist() == want
        xf = (xi.astype(np.float32) * np.float32(0.5))
        want = _brute_select([float(v) for v in xf], "f32", O.NONZERO)
        assert o.select_if(xf, O.NONZERO).tolist() == want


def pin_select_float_special_values(o):
    """IEEE != 0: -0.0 and +0.0 dropped, NaN, inf and denormals kept."""
    x = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1e-45, -1e-45, 2.5],
                 dtype=np.float32)
    got = o.select_if(x, O.NONZERO)
    assert got.shape[0] == 6
    assert np.isnan(got[0]) and got[1] == np.inf and got[2] == -np.inf
    assert got[3] > 0 and got[4] < 0 and got[5] == 2.5
    assert not o.pred_supported(O.F32, O.ODD) and not o.pred_supported(O.F32, O.EVEN)
    assert o.pred_supported(O.I32, O.ODD) and o.pred_supported(O.U32, O.EVEN)


def pin_select_negative_odd(o):
    """Odd by x & 1 in two's complement: -3 and -1 are odd, -2 is even."""
    x = np.array([-3, -2, -1, 0, 1, 2, 3, -2147483648, 2147483647], dtype=np.int32)
    assert o.select_if(x, O.ODD).tolist() == [-3, -1, 1, 3, 2147483647]
    assert o.select_if(x, O.EVEN).tolist() == [-2, 0, 2, -2147483648]


def pin_select_invariants(o):
    """count = sum of the predicate (numpy), output an order-preserving
    subsequence (the kept input positions, via numpy's boolean mask), all
    kept = copy, none kept = empty."""
    x = synth.remove_zeros(100_003, 1)
    got = o.select_if(x, O.NONZERO)
    mask = x != 0
    assert got.shape[0] == int(mask.sum()) == o.count_if(x, O.NONZERO)
    assert np.array_equal(got, x[np.flatnonzero(mask)])
    ones = np.ones(1000, dtype=np.int32)
    assert np.array_equal(o.select_if(ones, O.NONZERO), ones)
    assert o.select_if(np.zeros(1000, dtype=np.int32), O.NONZERO).shape[0] == 0
    odd = synth.uniform_i32(50_001, 3)
    assert np.array_equal(o.select_if(odd, O.ODD), odd[(odd & 1) == 1])


# ------------------------------------------------------------------ partition

def pin_partition_brute_force(o):
    """True element i goes to rank[i], false element i to T + i - rank[i]
    (the i - rank[i] identity of the Day 33 scatterPartition), O(n^2)."""
    rng = _rng(13)
    for n in [0, 1, 2, 5, 33, 64, 150]:
        x = rng.integers(-5, 6, size=n).astype(np.int32)
        for pred in (O.NONZERO, O.ODD, O.EVEN):
            keep = [_py_keep(int(v), "i32", pred) for v in x]
            T = sum(keep)
            want = [None] * n
            for i in range(n):
                rank = sum(1 for j in range(i) if keep[j])
                want[rank if keep[i] else T + i - rank] = int(x[i])
            got, t = o.partition(x, pred)
            assert t == T and got.tolist() == want, (n, pred)


def pin_partition_invariants(o):
    """Permutation of the input; first half = stable select, second half =
    stable select of the complement (numpy masks)."""
    x = synth.uniform_i32(200_001, 4)
    got, t = o.partition(x, O.EVEN)
    ev = (x & 1) == 0
    assert t == int(ev.sum())
    assert np.array_equal(np.sort(got), np.sort(x))
    assert np.array_equal(got[:t], x[ev]) and np.array_equal(got[t:], x[~ev])


# ------------------------------------------------------------------ radix

def pin_radix_matches_stable_argsort(o):
    """Full 32-bit sort = numpy stable argsort (a library routine): keys
    ascending, payload = original index, ties in input order."""
    keys, vals = synth.radix_keys(300_007, 5)
    keys[::7] = keys[3]  # plenty of ties
    ko, vo = o.split_radix(keys, vals)
    perm = np.argsort(keys, kind="stable")
    assert np.array_equal(ko, keys[perm]) and np.array_equal(vo, vals[perm])


def pin_radix_bit_ranges(o):
    """Bits [b, e): stable argsort of the key field (k >> b) & mask;
    a single bit equals the stable partition by 'bit clear'; an empty range
    copies; keys-only equals the keys of the keyed sort."""
    rng = _rng(14)
    keys = rng.integers(0, 2 ** 32, size=20_000, dtype=np.uint64).astype(np.uint32)
    vals = np.arange(keys.shape[0], dtype=np.uint32)
    for b, e in [(0, 1), (5, 6), (31, 32), (0, 8), (8, 24), (3, 3)]:
        field = (keys >> np.uint32(b)) & np.uint32((1 << (e - b)) - 1) if e > b else np.zeros_like(keys)
        perm = np.argsort(field, kind="stable")
        ko, vo = o.split_radix(keys, vals, b, e)
        assert np.array_equal(ko, keys[perm]) and np.array_equal(vo, perm.astype(np.uint32)), (b, e)
        ko2, vo2 = o.split_radix(keys, None, b, e)
        assert vo2 is None and np.array_equal(ko2, ko)
    b = 9
    clear = ((keys >> np.uint32(b)) & np.uint32(1)) == 0
    ko, _ = o.split_radix(keys, vals, b, b + 1)
    assert np.array_equal(ko, np.concatenate([keys[clear], keys[~clear]]))


def pin_radix_degenerate(o):
    """All-equal keys and already-sorted keys come back unchanged."""
    eq = np.full(4097, 12345, dtype=np.uint32)
    idx = np.arange(4097, dtype=np.uint32)
    ko, vo = o.split_radix(eq, idx)
    assert np.array_equal(ko, eq) and np.array_equal(vo, idx)
    srt = np.sort(synth.uniform_u32(4097, 77))
    ko, vo = o.split_radix(srt, idx)
    assert np.array_equal(ko, srt) and np.array_equal(vo, idx)


# ------------------------------------------------------------------ parameterised predicates

_NP_CMP = {O.LT: np.less, O.LE: np.less_equal, O.GT: np.greater, O.GE: np.greater_equal,
           O.EQ: np.equal, O.NE: np.not_equal}


def _cmp_inputs(rng, n):
    xi = rng.integers(-50, 51, size=n).astype(np.int32)
    xi[::17] = np.iinfo(np.int32).min
    xi[5::19] = np.iinfo(np.int32).max
    xu = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    xu[::13] = 7
    xf = (rng.standard_normal(n) * 3).astype(np.float32)
    specials = np.array([0.0, -0.0, np.nan, np.inf, -np.inf, 1e-45, -1e-45, 2.5], np.float32)
    xf[: 8 * (n // 64)] = np.tile(specials, n // 64)
    return xi, xu, xf


def pin_select_cmp_matches_numpy(o):
    """x OP v in the dtype's order equals numpy's element-wise comparison
    (IEEE for float32: NaN compares false except !=), for every operator."""
    rng = _rng(21)
    xi, xu, xf = _cmp_inputs(rng, 4096)
    cases = [(xi, [-50, -3, 0, 7, 2147483647, -2147483648]),
             (xu, [0, 7, 2 ** 31, 2 ** 32 - 1]),
             (xf, [0.0, -0.0, 2.5, float("inf"), float("nan"), -1e-45])]
    for x, values in cases:
        for v in values:
            for cmp, f in _NP_CMP.items():
                want = x[f(x, x.dtype.type(v))]
                got = o.select_if_cmp(x, cmp, v)
                assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (x.dtype, v, cmp)


def pin_select_mask_tests_match_numpy(o):
    """(bits & mask) == value and != value on the raw 32 bits, any dtype."""
    rng = _rng(22)
    xi, xu, xf = _cmp_inputs(rng, 4096)
    for x in (xi, xu, xf):
        b = x.view(np.uint32)
        for mask, value in [(1, 0), (1, 1), (0xF0, 0x30), (0x80000000, 0x80000000), (0, 0)]:
            sel = (b & np.uint32(mask)) == np.uint32(value)
            assert np.array_equal(o.select_if_cmp(x, O.MASK_EQ, value, mask).view(np.uint32), b[sel])
            assert np.array_equal(o.select_if_cmp(x, O.MASK_NE, value, mask).view(np.uint32), b[~sel])


def pin_fixed_predicates_are_special_cases(o):
    """ODD = mask 1 != 0, EVEN = mask 1 == 0, NONZERO = != 0 (float: IEEE)."""
    rng = _rng(23)
    xi, xu, xf = _cmp_inputs(rng, 2048)
    for x in (xi, xu):
        assert np.array_equal(o.select_if_cmp(x, O.MASK_NE, 0, 1), o.select_if(x, O.ODD))
        assert np.array_equal(o.select_if_cmp(x, O.MASK_EQ, 0, 1), o.select_if(x, O.EVEN))
        assert np.array_equal(o.select_if_cmp(x, O.NE, 0), o.select_if(x, O.NONZERO))
    assert np.array_equal(o.select_if_cmp(xf, O.NE, 0.0).view(np.uint32),
                          o.select_if(xf, O.NONZERO).view(np.uint32))


def pin_partition_cmp_invariants(o):
    """Kept half = numpy-selected elements in order, the rest after, stable."""
    rng = _rng(24)
    xi, xu, xf = _cmp_inputs(rng, 3000)
    for x, v, cmp in [(xi, 3, O.GE), (xu, 2 ** 31, O.LT), (xf, 0.0, O.GT), (xf, 1.0, O.NE)]:
        sel = _NP_CMP[cmp](x, x.dtype.type(v))
        got, t = o.partition_cmp(x, cmp, v)
        assert t == int(sel.sum())
        assert np.array_equal(got[:t].view(np.uint32), x[sel].view(np.uint32))
        assert np.array_equal(got[t:].view(np.uint32), x[~sel].view(np.uint32))


# ------------------------------------------------------------------ typed radix sort

def pin_radix_sort_int32_float32_match_argsort(o):
    """int32 and float32 keys (no NaN, no -0.0) sort as numpy's stable argsort;
    uint32 keys as the 32-bit one-bit-split sort."""
    rng = _rng(31)
    ki = rng.integers(-2 ** 31, 2 ** 31, size=50_001, dtype=np.int64).astype(np.int32)
    ki[::9] = ki[4]
    kf = (rng.standard_normal(50_001) * 1e3).astype(np.float32)
    kf[::7] = kf[3]
    kf[5::11] = np.float32(np.inf)
    kf[6::13] = np.float32(-np.inf)
    kf[kf == 0] = 1.0  # keep -0.0 out: numpy orders it equal to +0.0
    vals = np.arange(50_001, dtype=np.uint32)
    for k in (ki, kf):
        perm = np.argsort(k, kind="stable")
        ko, vo = o.radix_sort(k, vals)
        assert np.array_equal(ko.view(np.uint32), k[perm].view(np.uint32))
        assert np.array_equal(vo, perm.astype(np.uint32))
    ku = synth.uniform_u32(20_001, 6)
    ko, vo = o.radix_sort(ku, vals[:20_001])
    wk, wv = o.split_radix(ku, vals[:20_001])
    assert np.array_equal(ko, wk) and np.array_equal(vo, wv)


def pin_radix_sort_float_total_order(o):
    """IEEE 754 totalOrder: -NaN < -inf < -1 < -denormal < -0 < +0 < +denormal
    < 1 < +inf < +NaN, ties in input order."""
    order = [0xFFC00000, 0xFF800000, 0xBF800000, 0x80000001, 0x80000000, 0x00000000,
             0x00000001, 0x3F800000, 0x7F800000, 0x7FC00000]
    keys = np.array([order[i] for i in (7, 0, 5, 9, 4, 2, 8, 1, 6, 3, 5, 4)],
                    dtype=np.uint32).view(np.float32)
    ko, vo = o.radix_sort(keys, np.arange(12, dtype=np.uint32))
    want = [order[i] for i in (0, 1, 2, 3, 4, 4, 5, 5, 6, 7, 8, 9)]
    assert ko.view(np.uint32).tolist() == want
    assert vo.tolist() == [1, 7, 5, 9, 4, 11, 2, 10, 8, 0, 6, 3]


# ------------------------------------------------------------------ comparator helper

def pin_out_of_order_count(o):
    """countOutOfOrder counts positions that differ."""
    a = np.array([1, 2, 3, 4], dtype=np.int32)
    b = np.array([1, 3, 2, 4], dtype=np.int32)
    assert o.count_out_of_order(a, b) == 2 and o.count_out_of_order(a, a) == 0


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
# the cheap ones, for running against many mutants
FAST_PINS = [p for p in ALL_PINS if p not in (pin_scan_mod8_closed_form,
                                             pin_scan_every_fourth_two)]


def run(o, pins=None):
    """-> list of (pin name, message) for every pin that fails."""
    bad = []
    for p in pins or ALL_PINS:
        try:
            p(o)
        except (AssertionError, ValueError, IndexError, TypeError) as e:  # noqa: PERF203
            bad.append((p.__name__, repr(e)[:200]))
    return bad

