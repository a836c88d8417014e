"""The segmented-scan oracle against what fixes it from outside: every prefix
is a segmented reduction (the reduction oracle over that one prefix), numpy's
cumulative routines per segment, a Python brute force, closed forms; plus
planted mistakes the pins must catch."""
import functools
import os

import numpy as np
import pytest

import oracle
from oracle import brute

SRC = os.path.join(os.path.dirname(oracle.__file__), "scan_oracle.c")
KINDS = {"u32": np.uint32, "s32": np.int32, "f32": np.float32}


def _values(rng, kind, n):
    if kind == "f32":
        return (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 6, size=n)).astype(np.float32)
    if kind == "s32":
        return rng.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32)
    return rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)


def _offsets(rng, n, segs, start=0, stop=None):
    stop = n if stop is None else stop
    cuts = np.sort(rng.integers(start, stop + 1, size=segs - 1))
    return np.concatenate([[start], cuts, [stop]]).astype(np.int64)


def pin_prefix_is_reduction(scan):
    """out[r] (inclusive) is the reduction of values[offsets[s] .. r] by the
    reduction oracle; exclusive sum is the reduction of values[offsets[s] ..
    r - 1]; rows in no segment are 0."""
    rng = np.random.default_rng(1)
    for kind in KINDS:
        n = 150
        v = _values(rng, kind, n)
        off = _offsets(rng, n, 9, start=7, stop=140)
        for op, excl in (("sum", False), ("sum", True), ("min", False), ("max", False)):
            got = scan(v, off, op, excl)
            for s in range(len(off) - 1):
                for r in range(off[s], off[s + 1]):
                    end = r if excl else r + 1
                    if end == off[s]:
                        exp = np.zeros(1, v.dtype)
                    else:
                        exp = oracle.seg_reduce(v, np.array([off[s], end]), op, with_arg=False)
                    assert got[r].tobytes() == np.asarray(exp, v.dtype)[0].tobytes(), (kind, op, excl, r)
            outside = np.ones(n, bool)
            outside[off[0]:off[-1]] = False
            assert not np.any(got[outside]), (kind, op)


def pin_numpy_cumulative(scan):
    """Per segment: numpy cumsum (float64 for float32, then rounded; int64
    modulo 2^32 for integers), minimum / maximum.accumulate."""
    rng = np.random.default_rng(2)
    for kind in KINDS:
        n = 3000
        v = _values(rng, kind, n)
        off = _offsets(rng, n, 40)
        for op in ("sum", "min", "max"):
            got = scan(v, off, op, False)
            for s in range(len(off) - 1):
                seg = v[off[s]:off[s + 1]]
                if op == "sum":
                    if kind == "f32":
                        exp = np.cumsum(seg.astype(np.float64)).astype(np.float32)
                    else:
                        exp = (np.cumsum(seg.astype(np.int64)) % 2**32).astype(np.uint64).astype(np.uint32).view(v.dtype)
                else:
                    exp = (np.minimum if op == "min" else np.maximum).accumulate(seg)
                assert np.array_equal(got[off[s]:off[s + 1]].view(np.uint32), exp.view(np.uint32)), (kind, op, s)


def pin_brute_force(scan):
    """Equal to the Python brute force (each prefix reduced on its own)."""
    rng = np.random.default_rng(3)
    for trial in range(15):
        kind = ("u32", "s32", "f32")[trial % 3]
        n = int(rng.integers(0, 40))
        v = _values(rng, kind, n)
        off = _offsets(rng, n, int(rng.integers(1, 6)))
        for op, excl in (("sum", False), ("sum", True), ("min", False), ("max", False)):
            exp = np.array(brute.seg_scan(v.tolist(), off.tolist(), op, kind, excl), dtype=KINDS[kind])
            got = scan(v, off, op, excl)
            if kind == "f32" and op == "sum":
                # fsum (correctly rounded) against a double running sum: within a few ulps
                assert np.allclose(got, exp, rtol=1e-6, atol=1e-6), (trial, op, excl)
            else:
                assert np.array_equal(got, exp), (trial, op, excl)


def pin_closed_forms(scan):
    """Ones: inclusive sum = position in the segment + 1, exclusive = position;
    the exclusive sum of segment lengths over one segment is the offsets."""
    off = np.array([2, 2, 5, 9, 10], np.int64)
    ones = np.ones(12, np.int32)
    assert list(scan(ones, off, "sum", False)) == [0, 0, 1, 2, 3, 1, 2, 3, 4, 1, 0, 0]
    assert list(scan(ones, off, "sum", True)) == [0, 0, 0, 1, 2, 0, 1, 2, 3, 0, 0, 0]
    lengths = np.array([3, 0, 5, 1, 7], np.uint32)
    assert list(scan(lengths, np.array([0, 5]), "sum", True)) == [0, 3, 3, 8, 9]
    v = np.array([5, 3, 8, 1, 9], np.uint32)
    assert list(scan(v, np.array([0, 5]), "min", False)) == [5, 3, 3, 1, 1]
    assert list(scan(v, np.array([0, 5]), "max", False)) == [5, 5, 8, 8, 9]


ALL_PINS = [pin_prefix_is_reduction, pin_numpy_cumulative, pin_brute_force, pin_closed_forms]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_scan_oracle_pin(pin):
    pin(oracle.seg_scan)


def test_rejects():
    v = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle.seg_scan(v, np.array([0, 3, 2, 4]))
    with pytest.raises(ValueError):
        oracle.seg_scan(v, np.array([0, 4]), "max", exclusive=True)


MUTANTS = [
    ("no_reset_between_segments", [("        double dacc = 0.0;\n        uint32_t uacc = 0u;\n",
                                     ""),
                                    ("    for (int64_t s = 0; s < S; ++s) {\n        const int64_t b = offsets[s], e = offsets[s + 1];",
                                     "    double dacc = 0.0;\n    uint32_t uacc = 0u;\n    for (int64_t s = 0; s < S; ++s) {\n        const int64_t b = offsets[s], e = offsets[s + 1];")]),
    ("exclusive_as_inclusive", [("(float)(exclusive ? before : dacc)", "(float)dacc"),
                                ("exclusive ? before : uacc", "uacc")]),
    ("float_accumulator", [("double dacc = 0.0;", "float dacc = 0.0f;"), ("const double before = dacc;", "const float before = dacc;")]),
    ("outside_rows_kept", [("            ((uint32_t *)out)[r] = 0u;\n    }", "            ((uint32_t *)out)[r] = ((const uint32_t *)values)[r];\n    }")]),
    ("signed_as_unsigned", [("const int32_t x = ((const int32_t *)values)[r], y = ((int32_t *)out)[r - 1];",
                             "const uint32_t x = ((const uint32_t *)values)[r], y = ((uint32_t *)out)[r - 1];"),
                            ("((int32_t *)out)[r] = (op == SN_MIN ? x < y : x > y) ? x : y;",
                             "((uint32_t *)out)[r] = (op == SN_MIN ? x < y : x > y) ? x : y;")]),
    ("last_row_of_segment_dropped", [("for (int64_t r = b; r < e; ++r) {", "for (int64_t r = b; r + 1 < e; ++r) {")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_scan_mutant_is_caught(tmp_path, name, edits):
    mutated = open(SRC).read()
    for old, new in edits:
        assert old in mutated, f"mutation anchor for {name} not found"
        mutated = mutated.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.load_scan_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    scan = functools.partial(oracle.seg_scan, lib=lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(scan)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
