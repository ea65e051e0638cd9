"""The oracle against its pins, and the pins against planted mistakes.

CPU only.  The mutants are copies of oracle.c with one plausible mistake
each (a textual edit), compiled into a temporary directory; every mutant must
fail at least one pin, which shows that the pins can see that kind of error.
"""

import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, orc):
    pin(orc)


# (name, text in oracle.c, replacement) -- each a mistake someone could make
MUTANTS = [
    ("scan_inclusive_instead_of_exclusive",
     "        const uint32_t v = in[i];\n        out[i] = running;\n        running += v;",
     "        const uint32_t v = in[i];\n        running += v;\n        out[i] = running;"),
    ("scan_drops_last_term_of_total",
     "        running += v;\n    }\n    return running;",
     "        if (i + 1 < n) running += v;\n    }\n    return running;"),
    ("scan_f32_accumulates_in_float",
     "    double running = 0.0;\n    for (size_t i = 0; i < n; ++i) {\n        out[i] = running;",
     "    float running = 0.0f;\n    for (size_t i = 0; i < n; ++i) {\n        out[i] = running;"),
    ("scan_f32_off_by_one_index",
     "        out[i] = running;\n        running += (double)in[i];",
     "        out[i] = running;\n        running += (double)in[i + (i + 1 < n)];"),
    ("select_writes_wrong_slot",
     "        if (keep(in[i], dtype, pred)) {\n            out[m] = in[i];\n            ++m;",
     "        if (keep(in[i], dtype, pred)) {\n            out[m] = in[m];\n            ++m;"),
    ("odd_tests_wrong_bit",
     "    if (pred == ORC_ODD) return (bits & 1u) != 0u;",
     "    if (pred == ORC_ODD) return (bits & 2u) != 0u;"),
    ("float_nonzero_on_bits",
     "        if (dtype == ORC_F32) return bits_to_float(bits) != 0.0f;",
     "        if (dtype == ORC_F32) return bits != 0u;"),
    ("partition_second_half_restarts_at_zero",
     "    size_t second = first;\n    for (size_t i = 0; i < n; ++i) {\n        if (!keep(in[i], dtype, pred)) {",
     "    size_t second = 0;\n    for (size_t i = 0; i < n; ++i) {\n        if (!keep(in[i], dtype, pred)) {"),
    ("partition_second_half_reversed",
     "    size_t second = first;\n    for (size_t i = 0; i < n; ++i) {\n        if (!keep(in[i], dtype, pred)) {",
     "    size_t second = first;\n    for (size_t i = n; i-- > 0;) {\n        if (!keep(in[i], dtype, pred)) {"),
    ("split_set_bits_first",
     "        if (((keys[i] >> b) & 1u) == 0u) {\n            keys_out[zeros] = keys[i];",
     "        if (((keys[i] >> b) & 1u) != 0u) {\n            keys_out[zeros] = keys[i];"),
    ("split_uses_wrong_bit",
     "        split_by_bit(ka, va, kb, vb, n, b);",
     "        split_by_bit(ka, va, kb, vb, n, 31 - b);"),
    ("radix_skips_first_bit",
     "    for (int b = begin_bit; b < end_bit; ++b) {",
     "    for (int b = begin_bit + 1; b < end_bit; ++b) {"),
    ("cmp_le_as_lt_for_int",
     "        case ORC_LE: return x <= v;\n        case ORC_GT: return x > v;\n        case ORC_GE: return x >= v;\n        case ORC_EQ: return x == v;\n        default: return x != v;\n        }\n    }\n    switch",
     "        case ORC_LE: return x < v;\n        case ORC_GT: return x > v;\n        case ORC_GE: return x >= v;\n        case ORC_EQ: return x == v;\n        default: return x != v;\n        }\n    }\n    switch"),
    ("cmp_unsigned_order_for_int32",
     "    if (dtype == ORC_I32) {\n        int32_t x, v;",
     "    if (dtype == 99) {\n        int32_t x, v;"),
    ("cmp_mask_ignores_mask",
     "    if (cmp == ORC_MASK_EQ) return (bits & mask) == value;",
     "    if (cmp == ORC_MASK_EQ) return bits == value;"),
    ("float_key_positive_not_flipped",
     "    if (dtype == ORC_F32) return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);",
     "    if (dtype == ORC_F32) return (bits & 0x80000000u) ? ~bits : bits;"),
    ("int32_key_unsigned_order",
     "    if (dtype == ORC_I32) return bits ^ 0x80000000u;\n    if (dtype == ORC_F32) return (bits & 0x80000000u) ? ~bits",
     "    if (dtype == ORC_I32) return bits;\n    if (dtype == ORC_F32) return (bits & 0x80000000u) ? ~bits"),
    ("radix_drops_payload_swap",
     "        t = va; va = vb; vb = t;",
     "        (void)0;"),
    ("inclusive_scan_u32_stores_before_add",
     "        running += in[i];\n        out[i] = running;",
     "        out[i] = running;\n        running += in[i];"),
    ("inclusive_scan_f32_stores_before_add",
     "        running += (double)in[i];\n        out[i] = running;",
     "        out[i] = running;\n        running += (double)in[i];"),
    ("even_tests_wrong_bit",
     "    return (bits & 1u) == 0u; /* ORC_EVEN */",
     "    return (bits & 2u) == 0u; /* ORC_EVEN */"),
    ("int_nonzero_drops_negatives",
     "        return bits != 0u;\n    }",
     "        return (int32_t)bits > 0;\n    }"),
    ("count_if_skips_last_element",
     "    for (size_t i = 0; i < n; ++i) c += (size_t)keep(in[i], dtype, pred);",
     "    for (size_t i = 0; i + 1 < n; ++i) c += (size_t)keep(in[i], dtype, pred);"),
    ("float_key_negative_mapped_back_wrong",
     "    if (dtype == ORC_F32) return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;",
     "    if (dtype == ORC_F32) return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : (key ^ 0x80000000u);"),
]


# a mutant whose edit needs two sites lists the second one here
COMPANION = {
    "split_set_bits_first": ("        if (((keys[i] >> b) & 1u) != 0u) {\n            keys_out[ones] = keys[i];",
                             "        if (((keys[i] >> b) & 1u) == 0u) {\n            keys_out[ones] = keys[i];"),
}


def _compile(src_text, path):
    c = path.with_suffix(".c")
    c.write_text(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-w", "-o", str(path), str(c)],
                   check=True)


_CHILD = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins as P
bad = P.run(oracle.Oracle(oracle.load_library({so!r})), P.FAST_PINS)
print("FAILED_PINS", len(bad), [b[0] for b in bad])
"""


def _pins_in_child(so):
    """Run the fast pins against a build in a child process; a mutant may
    corrupt memory, and a crash counts as the mutant being caught."""
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _CHILD.format(root=os.path.dirname(tests), tests=tests, so=str(so))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return -1, r.stderr[-400:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED_PINS")][-1]
    return int(line.split()[1]), line


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = (oracle._SRC).read_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique in oracle.c"
    so = tmp_path / f"mut_{name}.so"
    mutated = src.replace(old, new)
    if name in COMPANION:
        a, b = COMPANION[name]
        assert mutated.count(a) == 1
        mutated = mutated.replace(a, b)
    _compile(mutated, so)
    nbad, info = _pins_in_child(so)
    assert nbad != 0, f"no pin noticed the planted mistake {name}: {info}"


def test_unmutated_copy_passes(tmp_path):
    so = tmp_path / "copy.so"
    _compile(oracle._SRC.read_text(), so)
    nbad, info = _pins_in_child(so)
    assert nbad == 0, info
