"""The RLE / offsets-producer oracle against what the pages and plain facts
fix, and against an independent brute force; plus planted mistakes that the
pins must catch."""
import functools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SRC = os.path.join(os.path.dirname(oracle.__file__), "rle_oracle.c")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# ---- pins: each takes an rle(keys) -> (values, lengths, offsets) callable --------------

def pin_printed_example(rle):
    """GPURunLengthEncode, 'What is run-length encoding?' / 'Why RLE matters':
    the printed input, its values, lengths and offsets."""
    g = _golden("luma_run_length_example.json")
    v, l, o = rle(np.array(g["input"], np.uint32))
    assert list(v) == g["run_values"] and list(l) == g["run_lengths"] and list(o) == g["offsets"]


def pin_adjacency_not_uniqueness(rle):
    """The same page: runs are adjacent equal values, not global uniqueness."""
    g = _golden("luma_rle_adjacency_example.json")
    v, l, o = rle(np.array(g["input"], np.uint32))
    assert list(v) == g["run_values"]
    assert list(l) == [2, 1, 1] and list(o) == [0, 2, 3, 4]


def pin_empty_input(rle):
    """'Contract': empty input writes count = 0."""
    v, l, o = rle(np.zeros(0, np.uint32))
    assert len(v) == 0 and len(l) == 0 and list(o) == [0]


def pin_closed_forms(rle):
    """All equal: one run of length n.  All distinct: n runs of length 1.
    Extreme values compare as unsigned 32-bit integers."""
    n = 1000
    v, l, o = rle(np.full(n, 7, np.uint32))
    assert list(v) == [7] and list(l) == [n] and list(o) == [0, n]
    keys = np.arange(n, dtype=np.uint32)
    v, l, o = rle(keys)
    assert np.array_equal(v, keys) and (l == 1).all() and np.array_equal(o, np.arange(n + 1))
    keys = np.array([0xFFFFFFFF, 0xFFFFFFFF, 0, 0x80000000, 0x80000000, 0x7FFFFFFF], np.uint32)
    v, l, o = rle(keys)
    assert list(v) == [0xFFFFFFFF, 0, 0x80000000, 0x7FFFFFFF] and list(l) == [2, 1, 2, 1]


def pin_invariants_and_brute_force(rle):
    """On random keys: equal to the groupby brute force, lengths sum to n,
    values[r] == keys[offsets[r]], adjacent runs differ, every length >= 1."""
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(0, 300))
        keys = np.repeat(rng.integers(0, 5, size=n).astype(np.uint32), rng.integers(1, 4, size=n))[:n]
        v, l, o = rle(keys)
        bv, bl, bo = brute.rle(keys.tolist())
        assert list(v) == bv and list(l) == bl and list(o) == bo, trial
        assert int(l.sum()) == n and (l >= 1).all()
        if len(v):
            assert np.array_equal(v, keys[o[:-1]])
            assert (v[1:] != v[:-1]).all()


def pin_composition_with_reduction(rle):
    """'Composition': RLE offsets delimit the runs for the segmented reduction,
    so each run's min and max are its value and its sum is value x length."""
    rng = np.random.default_rng(11)
    keys = np.sort(rng.integers(0, 50, size=2000).astype(np.uint32))
    v, l, o = rle(keys)
    mn, amn = oracle.seg_reduce(keys, o, "min")
    mx, amx = oracle.seg_reduce(keys, o, "max")
    sm = oracle.seg_reduce(keys, o, "sum")
    assert np.array_equal(mn, v) and np.array_equal(mx, v) and np.array_equal(amn, o[:-1])
    assert np.array_equal(sm, (v.astype(np.uint64) * l).astype(np.uint32))


ALL_PINS = [pin_printed_example, pin_adjacency_not_uniqueness, pin_empty_input, pin_closed_forms,
            pin_invariants_and_brute_force, pin_composition_with_reduction]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_rle_oracle_pin(pin):
    pin(oracle.rle)


def test_flags_to_offsets_oracle():
    """GPUSegmentedLayout: offsets are the flagged indices, then n; checked
    against the brute force, and against RLE boundary flags."""
    rng = np.random.default_rng(3)
    for trial in range(40):
        n = int(rng.integers(0, 200))
        flags = (rng.random(n) < rng.random()).astype(np.uint8) * rng.integers(1, 255, size=n).astype(np.uint8)
        assert list(oracle.flags_to_offsets(flags)) == brute.flags_to_offsets(flags.tolist()), trial
    assert list(oracle.flags_to_offsets(np.zeros(5, np.uint8))) == [5]
    assert list(oracle.flags_to_offsets(np.ones(4, np.uint8))) == [0, 1, 2, 3, 4]
    keys = np.array([2, 2, 2, 5, 5, 9, 9, 9, 9], np.uint32)
    boundary = np.r_[1, keys[1:] != keys[:-1]].astype(np.uint8)
    assert list(oracle.flags_to_offsets(boundary)) == list(oracle.rle(keys)[2])


MUTANTS = [
    ("length_off_by_one", [("lengths[runs] = (uint32_t)(i - start);", "lengths[runs] = (uint32_t)(i - start + 1);")]),
    ("last_run_dropped", [("int ends_here = i > 0 && (i == n || keys[i] != keys[i - 1]);",
                           "int ends_here = i > 0 && i < n && keys[i] != keys[i - 1];")]),
    ("runs_only_on_increase", [("keys[i] != keys[i - 1]", "keys[i] > keys[i - 1]")]),
    ("value_from_next_run", [("values[runs] = keys[start];", "values[runs] = keys[i < n ? i : start];")]),
    ("offsets_end_missing", [("        offsets[runs] = n;", "        offsets[runs] = n - 1;")]),
    ("signed_compare", [("keys[i] != keys[i - 1]", "(int32_t)keys[i] / 2 != (int32_t)keys[i - 1] / 2")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_rle_mutant_is_caught(tmp_path, name, edits):
    mutated = open(SRC).read()
    for old, new in edits:
        assert old in mutated, f"mutation anchor for {name} not found"
        mutated = mutated.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.load_rle_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    rle = functools.partial(oracle.rle, lib=lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(rle)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
