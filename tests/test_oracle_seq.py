"""The input-order float32 oracle (graph-reduce README, "Correctness": a fixed
summation order, bitwise equal to torch.segment_reduce) against what the
definition and IEEE float32 arithmetic fix, against an independent numpy
float32 brute force, and planted mistakes that the pins must catch."""
import functools
import os

import numpy as np
import pytest

import oracle
from oracle import brute

SRC = os.path.join(os.path.dirname(oracle.__file__), "seq_oracle.c")
F32 = np.float32


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


# ---- pins: each takes a seq(values, offsets, op) callable -----------------------------

def pin_exact_small_integers(seq):
    """Sums of small integers are exact in float32 in any order: the result is
    the integer sum; the mean is the correctly rounded quotient."""
    rng = np.random.default_rng(1)
    v = rng.integers(-1000, 1000, size=500).astype(np.float32)
    off = np.array([0, 1, 7, 7, 100, 333, 500], np.int64)
    got = seq(v, off, "sum")
    exp = [float(sum(int(x) for x in v[off[i]:off[i + 1]])) for i in range(len(off) - 1)]
    assert list(got) == exp
    m = seq(v, off, "mean")
    for i in range(len(off) - 1):
        n = off[i + 1] - off[i]
        assert m[i] == (F32(exp[i]) / F32(n) if n else F32(0))


def pin_input_order(seq):
    """Order-sensitive float32 cases (spacing of float32 at 1e8 is 8):
    - [1e8, -1e8, 1]: 0 then 1 -> 1;
    - [1e8, 1, -1e8, 1]: 1e8 + 1 rounds to 1e8, so 0, then 1 -> 1 (a pairwise
      tree gives (1e8 + 1) + (-1e8 + 1) = 0, the exact sum is 2);
    - [1, -1e8, 1e8]: -1e8 + 1e8 -> 0 (the reverse order gives 1)."""
    v = np.array([1e8, -1e8, 1, 1e8, 1, -1e8, 1, 1, -1e8, 1e8], np.float32)
    off = np.array([0, 3, 7, 10], np.int64)
    got = seq(v, off, "sum")
    assert list(got) == [1.0, 1.0, 0.0]


def pin_fold_starts_at_zero(seq):
    """The fold starts from +0.0: a segment holding only -0.0 sums to +0.0,
    and an empty segment gives 0 for sum and mean."""
    v = np.array([-0.0, -0.0, -0.0], np.float32)
    off = np.array([0, 1, 3, 3], np.int64)
    got = seq(v, off, "sum")
    assert list(_bits(got)) == [0, 0, 0]
    assert list(_bits(seq(v, off, "mean"))) == [0, 0, 0]


def pin_columns_independent(seq):
    """[N, F]: column f of the result is the 1-D result of column f."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal((300, 5)).astype(np.float32) * np.float32(1e3)
    off = np.array([0, 2, 2, 150, 151, 300], np.int64)
    got = seq(v, off, "sum")
    for f in range(5):
        assert np.array_equal(_bits(got[:, f]), _bits(seq(np.ascontiguousarray(v[:, f]), off, "sum")))


def pin_brute_force(seq):
    """Bitwise equal to the numpy float32 loop on random inputs with wide
    magnitudes (so that the order of additions shows in the bits)."""
    rng = np.random.default_rng(3)
    for trial in range(25):
        n = int(rng.integers(0, 120))
        feat = int(rng.integers(1, 4))
        v = (rng.standard_normal((n, feat)) * 10.0 ** rng.integers(-3, 8, size=(n, feat))).astype(np.float32)
        cuts = np.sort(rng.integers(0, n + 1, size=int(rng.integers(0, 12))))
        off = np.concatenate([[0], cuts, [n]]).astype(np.int64)
        for op in ("sum", "mean"):
            got = seq(v, off, op)
            exp = brute.seg_reduce_sequential(v, off, op)
            assert np.array_equal(_bits(got), _bits(exp)), (trial, op)


ALL_PINS = [pin_exact_small_integers, pin_input_order, pin_fold_starts_at_zero,
            pin_columns_independent, pin_brute_force]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_sequential_oracle_pin(pin):
    pin(oracle.seg_reduce_sequential)


def test_brute_force_is_itself_order_sensitive():
    """The brute force keeps float32 rounding per addition: it gives 1 where
    the exact sum is 2."""
    import math
    v = np.array([1e8, 1, -1e8, 1], np.float32)
    assert brute.seg_reduce_sequential(v, [0, 4])[0] == 1.0
    assert math.fsum(float(x) for x in v) == 2.0


def test_matches_torch_segment_reduce_on_the_cpu():
    """graph-reduce README, "Correctness": the fixed-order CSR sum is bitwise
    equal to torch.segment_reduce.  torch's CPU segment_reduce is an
    implementation of the same definition written by others: the oracle
    must agree with it bit for bit, for [N] and [N, F], sum and mean."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    for shape, segs in (((4000,), 300), ((3000, 5), 200), ((2000, 64), 50)):
        v = (rng.standard_normal(shape) * 10.0 ** rng.integers(-3, 8, size=shape)).astype(np.float32)
        cuts = np.sort(rng.integers(0, shape[0] + 1, size=segs - 1))
        off = np.concatenate([[0], cuts, [shape[0]]]).astype(np.int64)
        for op in ("sum", "mean"):
            exp = torch.segment_reduce(torch.from_numpy(v), op, offsets=torch.from_numpy(off),
                                       axis=0, unsafe=True).numpy()
            got = oracle.seg_reduce_sequential(v, off, op)
            nonempty = np.diff(off) > 0
            # torch's mean of an empty segment is NaN; the pages' (and this mode's) is 0
            assert np.array_equal(got[nonempty].view(np.uint32), exp[nonempty].view(np.uint32)), (shape, op)


def test_rejects_bad_offsets_and_ops():
    v = np.zeros(4, np.float32)
    with pytest.raises(ValueError):
        oracle.seg_reduce_sequential(v, np.array([0, 3, 2, 4]), "sum")
    with pytest.raises(ValueError):
        oracle.seg_reduce_sequential(v, np.array([0, 5]), "sum")
    with pytest.raises(ValueError):
        oracle.seg_reduce_sequential(v, np.array([0, 4]), "max")


MUTANTS = [
    ("reverse_order", [("for (int64_t r = b; r < e; ++r)\n                acc = acc + values[r * F + f];",
                        "for (int64_t r = e - 1; r >= b; --r)\n                acc = acc + values[r * F + f];")]),
    ("double_accumulator", [("float acc = 0.0f;", "double acc = 0.0;"),
                            ("out[s * F + f] = acc;", "out[s * F + f] = (float)acc;"),
                            ("acc = e > b ? acc / (float)(e - b) : 0.0f;", "acc = e > b ? acc / (double)(e - b) : 0.0;")]),
    ("pairwise_halves", [("for (int64_t r = b; r < e; ++r)\n                acc = acc + values[r * F + f];",
                          "float a1 = 0.0f, a2 = 0.0f;\n            for (int64_t r = b; r < e; ++r) {\n"
                          "                if (r < b + (e - b) / 2) a1 = a1 + values[r * F + f];\n"
                          "                else a2 = a2 + values[r * F + f]; }\n            acc = a1 + a2;")]),
    ("starts_at_first_row", [("float acc = 0.0f;\n            for (int64_t r = b; r < e; ++r)",
                              "float acc = e > b ? values[b * F + f] : 0.0f;\n            for (int64_t r = b + 1; r < e; ++r)")]),
    ("mean_by_length_plus_one", [("acc / (float)(e - b)", "acc / (float)(e - b + 1)")]),
    ("column_stride_wrong", [("acc = acc + values[r * F + f];", "acc = acc + values[r + f * N];")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_sequential_mutant_is_caught(tmp_path, name, edits):
    mutated = open(SRC).read()
    for old, new in edits:
        assert old in mutated, f"mutation anchor for {name} not found"
        mutated = mutated.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.load_seq_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    seq = functools.partial(oracle.seg_reduce_sequential, lib=lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(seq)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
