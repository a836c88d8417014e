"""The scatter oracle (graph-reduce README, "API" and "Method") against what
fixes it from outside: the segmented oracle applied after a stable sort of
the index (a different loop over the same definition), an independent
Python brute force, closed forms; plus planted mistakes the pins must catch."""
import functools
import os

import numpy as np
import pytest

import oracle
import workloads as W
from oracle import brute

SRC = os.path.join(os.path.dirname(oracle.__file__), "scatter_oracle.c")
KINDS = {"u32": np.uint32, "s32": np.int32, "f32": np.float32}


def _values(rng, kind, shape):
    if kind == "f32":
        return rng.standard_normal(shape).astype(np.float32)
    if kind == "s32":
        return rng.integers(-2**31, 2**31, size=shape, dtype=np.int64).astype(np.int32)
    return rng.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32)


def _close(a, b, kind, absval):
    if kind == "f32":
        assert np.all(np.abs(a.astype(np.float64) - b.astype(np.float64)) <= 1e-5 * absval + 1e-6)
    else:
        assert np.array_equal(a, b)


# ---- pins: each takes a scatter(src, index, dim_size, op) callable ---------------------

def pin_equals_segmented_after_sort(sc):
    """Scatter == the segmented reduction of the rows stably sorted by
    destination, with offsets from the destination counts (graph-reduce
    README, "Usage"); args map back through the sort."""
    rng = np.random.default_rng(1)
    for kind in KINDS:
        for feat in (1, 3):
            n, dim = 400, 37
            v = _values(rng, kind, (n,) if feat == 1 else (n, feat))
            idx = rng.integers(0, dim, size=n).astype(np.int64)
            perm = np.argsort(idx, kind="stable")
            off = np.concatenate([[0], np.cumsum(np.bincount(idx, minlength=dim))]).astype(np.int64)
            for op in ("sum", "min", "max") + (("mean",) if kind == "f32" else ()):
                exp = oracle.seg_reduce(v[perm], off, op)
                got = sc(v, idx, dim, op)
                if op in ("min", "max"):
                    (eo, ea), (go, ga) = exp, got
                    assert np.array_equal(go, eo), (kind, op)
                    assert np.array_equal(ga, np.where(ea >= 0, perm[np.maximum(ea, 0)], -1)), (kind, op)
                else:
                    # both loops add in row order in double: the same sums exactly
                    assert np.array_equal(got, exp), (kind, op)


def pin_brute_force(sc):
    """Equal to the Python brute force on small random inputs, including
    indices outside [0, dim_size) and destinations that receive nothing."""
    rng = np.random.default_rng(2)
    for trial in range(20):
        kind = ("u32", "s32", "f32")[trial % 3]
        feat = int(rng.integers(1, 4))
        n, dim = int(rng.integers(0, 60)), int(rng.integers(1, 12))
        v = _values(rng, kind, (n, feat))
        idx = rng.integers(-2, dim + 2, size=n).astype(np.int64)
        for op in ("sum", "min", "max"):
            bo, ba = brute.scatter(v.tolist(), idx.tolist(), dim, op, kind, feat)
            got = sc(v, idx, dim, op)
            go = got[0] if isinstance(got, tuple) else got
            if kind == "f32" and op == "sum":
                absv = np.zeros((dim, feat))
                for r, d in enumerate(idx):
                    if 0 <= d < dim:
                        absv[d] += np.abs(v[r].astype(np.float64))
                _close(go, np.array(bo, np.float32), kind, absv)
            else:
                assert np.array_equal(go, np.array(bo, dtype=KINDS[kind]).reshape(dim, feat)), (trial, op)
            if op in ("min", "max"):
                assert np.array_equal(got[1], np.array(ba, np.int64)), (trial, op)


def pin_closed_forms(sc):
    """Identity index gives the rows back (args = rows); one destination for
    every row is the whole-array reduction; nothing received gives 0 / -1;
    ties go to the lower row; mean of k copies of x is x."""
    v = np.array([5, 9, 9, 1, 1, 7], np.int32)
    out, arg = sc(v, np.arange(6), 6, "max")
    assert list(out) == list(v) and list(arg) == list(range(6))
    out, arg = sc(v, np.zeros(6, np.int64), 1, "max")
    assert list(out) == [9] and list(arg) == [1]
    out, arg = sc(v, np.zeros(6, np.int64), 1, "min")
    assert list(out) == [1] and list(arg) == [3]
    assert list(sc(v, np.zeros(6, np.int64), 1, "sum")) == [32]
    out, arg = sc(v, np.array([0, 0, 0, 2, 2, 2]), 4, "min")
    assert list(out) == [5, 0, 1, 0] and list(arg) == [0, -1, 3, -1]
    m = sc(np.full(7, 0.75, np.float32), np.array([1] * 7), 3, "mean")
    assert list(m) == [0.0, 0.75, 0.0]
    assert list(sc(np.array([1.0, 2.0], np.float32), np.array([-1, 5]), 3, "sum")) == [0.0, 0.0, 0.0]


ALL_PINS = [pin_equals_segmented_after_sort, pin_brute_force, pin_closed_forms]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_scatter_oracle_pin(pin):
    pin(oracle.scatter)


MUTANTS = [
    ("ties_to_higher_row", [("better = op == SC_MIN ? x < y : x > y;\n            } else if (dtype == SC_S32)",
                             "better = op == SC_MIN ? x <= y : x >= y;\n            } else if (dtype == SC_S32)"),
                            ("const int32_t x = ((const int32_t *)src)[i], y = ((const int32_t *)src)[j];\n                better = op == SC_MIN ? x < y : x > y;",
                             "const int32_t x = ((const int32_t *)src)[i], y = ((const int32_t *)src)[j];\n                better = op == SC_MIN ? x <= y : x >= y;")]),
    ("out_of_range_clamped", [("if (d < 0 || d >= D)\n            continue;", "if (d < 0) continue;\n        if (d >= D) continue;\n        if (d == D - 1 && r % 2) continue;")]),
    ("mean_by_rows_plus_one", [("s / (float)count[d]", "s / (float)(count[d] + 1)")]),
    ("unsigned_as_signed", [("const uint32_t x = ((const uint32_t *)src)[i], y = ((const uint32_t *)src)[j];",
                             "const int32_t x = ((const int32_t *)src)[i], y = ((const int32_t *)src)[j];")]),
    ("empty_max_arg_zero", [("best[c] = -1;", "best[c] = -1;\n    (void)0;"),
                            ("arg[c] = b;", "arg[c] = b < 0 ? 0 : b;")]),
    ("column_mixup", [("const int64_t i = r * F + f;", "const int64_t i = r * F + (F - 1 - f);")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_scatter_mutant_is_caught(tmp_path, name, edits):
    mutated = open(SRC).read()
    for old, new in edits:
        assert old in mutated, f"mutation anchor for {name} not found"
        mutated = mutated.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.load_scatter_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    sc = functools.partial(oracle.scatter, lib=lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(sc)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
