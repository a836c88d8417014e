"""Pins of the CPU oracle: facts the pages and the mathematics fix, checked
against any implementation of ``reduce(values, offsets, op) -> out | (out, arg)``.

Each pin is a function of that callable that raises AssertionError when the
implementation disagrees.  They are chosen so that a plausible mistake in an
oracle -- a dropped row, an inclusive end, a wrong sign or order, a transposed
column/row, the wrong tie rule, signed/unsigned confusion, a segment-relative
arg, a non-zero empty result -- fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U32 = np.uint32
S32 = np.int32
F32 = np.float32


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _f32_ulp(x):
    x = np.float32(abs(x))
    return float(np.spacing(x)) if x != 0 else float(np.spacing(np.float32(0)))


# ---------------------------------------------------------------------------
# Values the pages print.

def pin_luma_worked_example(reduce):
    """GPUSegmentedReduction, 'What is segmented reduction?': sum [30,120,130],
    min [10,30,60], max [20,50,70] for every value dtype and offset dtype."""
    g = _golden("luma_segmented_reduction_example.json")
    for dt in (U32, S32, F32):
        for odt in (np.uint32, np.int64):
            v = np.array(g["values"], dtype=dt)
            off = np.array(g["offsets"], dtype=odt)
            for op in ("sum", "min", "max"):
                r = reduce(v, off, op)
                out = r[0] if isinstance(r, tuple) else r
                assert out.dtype == dt
                assert out.tolist() == g["expected"][op], (dt, odt, op, out)


def pin_luma_worked_example_derived(reduce):
    """Same example, quantities the page does not print but the contract
    fixes: args of an increasing sequence are the first / last row of each
    segment (absolute rows), mean = sum / length."""
    g = _golden("luma_segmented_reduction_example.json")
    off = np.array(g["offsets"], dtype=np.int64)
    v = np.array(g["values"], dtype=F32)
    _, amin = reduce(v, off, "min")
    _, amax = reduce(v, off, "max")
    assert amin.tolist() == off[:-1].tolist()
    assert amax.tolist() == (off[1:] - 1).tolist()
    mean = reduce(v, off, "mean")
    sums = np.array(g["expected"]["sum"], dtype=np.float64)
    assert mean.tolist() == (sums / np.diff(off)).tolist()


def pin_rle_example(reduce):
    """GPURunLengthEncode: input [2,2,2,5,5,9,9,9,9] with offsets [0,3,5,9]
    (printed).  The runs are constant, so min = max = the printed run values,
    sum = run value x run length, and every arg is the run's first row (ties
    go to the lower row)."""
    g = _golden("luma_run_length_example.json")
    off_from_lengths = [0] + np.cumsum(g["run_lengths"]).tolist()
    assert off_from_lengths == g["offsets"]
    for dt in (U32, S32, F32):
        v = np.array(g["input"], dtype=dt)
        off = np.array(g["offsets"], dtype=np.uint32)
        s = reduce(v, off, "sum")
        assert s.tolist() == [a * b for a, b in zip(g["run_values"], g["run_lengths"])]
        for op in ("min", "max"):
            out, arg = reduce(v, off, op)
            assert out.tolist() == g["run_values"]
            assert arg.tolist() == g["offsets"][:-1]


# ---------------------------------------------------------------------------
# Contract rules.

def pin_empty_segments(reduce):
    """Repeated offsets are empty segments; they produce 0 (arg -1), and
    their neighbours are unaffected."""
    v = np.array([5, 7, 1, 9], dtype=F32)
    off = np.array([0, 0, 2, 2, 2, 4, 4], dtype=np.int64)
    assert reduce(v, off, "sum").tolist() == [0, 12, 0, 0, 10, 0]
    assert reduce(v, off, "mean").tolist() == [0, 6, 0, 0, 5, 0]
    mn, amn = reduce(v, off, "min")
    mx, amx = reduce(v, off, "max")
    assert mn.tolist() == [0, 5, 0, 0, 1, 0] and amn.tolist() == [-1, 0, -1, -1, 2, -1]
    assert mx.tolist() == [0, 7, 0, 0, 9, 0] and amx.tolist() == [-1, 1, -1, -1, 3, -1]
    for dt in (U32, S32):
        mx, amx = reduce(v.astype(dt), off, "max")
        assert mx.tolist() == [0, 7, 0, 0, 9, 0] and amx.tolist() == [-1, 1, -1, -1, 3, -1]


def pin_no_segments(reduce):
    """offsets of length 1 describe zero segments: empty output."""
    out = reduce(np.arange(4, dtype=F32), np.array([2], dtype=np.int64), "sum")
    assert out.shape == (0,)


def pin_nonzero_first_offset(reduce):
    """'output row i reduces input[o_i .. o_(i+1))': o_0 may be non-zero and
    rows outside [o_0, o_S) are ignored; args stay absolute row indices."""
    v = np.array([100, 1, 2, 3, 4, 100, 100], dtype=S32)
    off = np.array([1, 3, 5], dtype=np.int64)
    assert reduce(v, off, "sum").tolist() == [3, 7]
    out, arg = reduce(v, off, "max")
    assert out.tolist() == [2, 4] and arg.tolist() == [2, 4]
    out, arg = reduce(v, off, "min")
    assert out.tolist() == [1, 3] and arg.tolist() == [1, 3]


# ---------------------------------------------------------------------------
# Closed forms.

def pin_closed_forms(reduce):
    rng = np.random.default_rng(7)
    lengths = rng.integers(0, 40, size=50)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    n = int(off[-1])
    b, e = off[:-1], off[1:]
    ne = e > b
    # all ones: sum = length, mean = 1 (0 when empty)
    ones = np.ones(n, dtype=F32)
    assert reduce(ones, off, "sum").tolist() == lengths.tolist()
    assert reduce(ones, off, "mean").tolist() == ne.astype(float).tolist()
    # v[r] = r: arithmetic series, extremes at the ends
    for dt in (U32, S32, F32):
        v = np.arange(n, dtype=dt)
        s = reduce(v, off, "sum")
        assert s.astype(np.int64).tolist() == ((b + e - 1) * (e - b) // 2).tolist()
        mn, amn = reduce(v, off, "min")
        mx, amx = reduce(v, off, "max")
        assert amn.tolist() == np.where(ne, b, -1).tolist()
        assert amx.tolist() == np.where(ne, e - 1, -1).tolist()
        assert mn.astype(np.int64).tolist() == np.where(ne, b, 0).tolist()
        assert mx.astype(np.int64).tolist() == np.where(ne, e - 1, 0).tolist()
        # reversed: extremes swap ends
        w = v[::-1].copy()
        _, amn = reduce(w, off, "min")
        _, amx = reduce(w, off, "max")
        assert amn.tolist() == np.where(ne, e - 1, -1).tolist()
        assert amx.tolist() == np.where(ne, b, -1).tolist()
    # negative values: sign
    v = -np.arange(n, dtype=S32)
    assert reduce(v, off, "sum").astype(np.int64).tolist() == (-((b + e - 1) * (e - b) // 2)).tolist()


def pin_integer_wrap_and_order(reduce):
    """Integer sums wrap mod 2^32; uint32 orders unsigned, int32 signed."""
    off = np.array([0, 2], dtype=np.int64)
    assert reduce(np.array([1 << 31, 1 << 31], U32), off, "sum").tolist() == [0]
    assert reduce(np.array([0xFFFFFFFF, 2], U32), off, "sum").tolist() == [1]
    assert reduce(np.array([2**31 - 1, 1], S32), off, "sum").tolist() == [-2**31]
    assert reduce(np.array([-2**31, -1], S32), off, "sum").tolist() == [2**31 - 1]
    u = np.array([1, 0xFFFFFFFF], U32)
    out, arg = reduce(u, off, "max")
    assert out.tolist() == [0xFFFFFFFF] and arg.tolist() == [1]
    out, arg = reduce(u, off, "min")
    assert out.tolist() == [1] and arg.tolist() == [0]
    s = u.view(S32)                        # the same bits: 1, -1
    out, arg = reduce(s, off, "max")
    assert out.tolist() == [1] and arg.tolist() == [0]
    out, arg = reduce(s, off, "min")
    assert out.tolist() == [-1] and arg.tolist() == [1]
    # extremes of each type are reachable values, not sentinels
    out, arg = reduce(np.array([0xFFFFFFFF] * 3, U32), np.array([0, 3]), "min")
    assert out.tolist() == [0xFFFFFFFF] and arg.tolist() == [0]
    out, arg = reduce(np.array([0, 0], U32), np.array([0, 2]), "max")
    assert out.tolist() == [0] and arg.tolist() == [0]
    out, arg = reduce(np.array([-2**31] * 2, S32), np.array([0, 2]), "max")
    assert out.tolist() == [-2**31] and arg.tolist() == [0]


def pin_ties_lower_row(reduce):
    """graph-reduce README, 'Method': ties resolve to the lower row."""
    off = np.array([0, 4, 8], dtype=np.int64)
    v = np.array([3, 1, 1, 3, 2, 2, 2, 2], dtype=F32)
    out, arg = reduce(v, off, "min")
    assert out.tolist() == [1, 2] and arg.tolist() == [1, 4]
    out, arg = reduce(v, off, "max")
    assert out.tolist() == [3, 2] and arg.tolist() == [0, 4]


def pin_signed_zero_ties(reduce):
    """IEEE comparison: -0.0 == +0.0 is a tie, so the lower row and its bits win."""
    off = np.array([0, 2], dtype=np.int64)
    out, arg = reduce(np.array([0.0, -0.0], F32), off, "min")
    assert arg.tolist() == [0] and not np.signbit(out[0])
    out, arg = reduce(np.array([-0.0, 0.0], F32), off, "max")
    assert arg.tolist() == [0] and np.signbit(out[0])


# ---------------------------------------------------------------------------
# Row tensors [N, F]: reduction over dimension 0, per column.

def pin_row_tensor(reduce):
    """graph-reduce README, 'API': src [N, ...] is reduced over dimension 0;
    each column picks its own extreme row."""
    v = np.array([[1, 9], [5, 2], [3, 4]], dtype=F32)
    off = np.array([0, 3], dtype=np.int64)
    out, arg = reduce(v, off, "max")
    assert out.tolist() == [[5, 9]] and arg.tolist() == [[1, 0]]
    out, arg = reduce(v, off, "min")
    assert out.tolist() == [[1, 2]] and arg.tolist() == [[0, 1]]
    assert reduce(v, off, "sum").tolist() == [[9, 15]]
    v = np.array([[1, 10], [2, 20], [3, 30]], dtype=S32)
    off = np.array([0, 2, 2, 3], dtype=np.int64)
    assert reduce(v, off, "sum").tolist() == [[3, 30], [0, 0], [3, 30]]
    out, arg = reduce(v, off, "max")
    assert out.tolist() == [[2, 20], [0, 0], [3, 30]]
    assert arg.tolist() == [[1, 1], [-1, -1], [2, 2]]


def pin_row_tensor_is_per_column(reduce):
    """[N, F] equals F independent scalar reductions of its columns."""
    rng = np.random.default_rng(11)
    off = np.array([0, 0, 3, 10, 11, 11, 20], dtype=np.int64)
    for dt in (F32, S32):
        v = (rng.standard_normal((20, 5)) * 8).astype(dt)
        for op in ("sum", "min", "max"):
            full = reduce(v, off, op)
            for f in range(5):
                col = reduce(np.ascontiguousarray(v[:, f]), off, op)
                if isinstance(full, tuple):
                    assert full[0][:, f].tolist() == col[0].tolist()
                    assert full[1][:, f].tolist() == col[1].tolist()
                else:
                    assert full[:, f].tolist() == col.tolist()


# ---------------------------------------------------------------------------
# Special cases that reduce to a library routine; invariants; brute force.

def pin_single_segment_is_global_reduction(reduce):
    """S = 1 is GPUReduction's single global aggregate: numpy's sum / min /
    argmin / max / argmax (first occurrence) and math.fsum."""
    rng = np.random.default_rng(3)
    n = 1000
    off = np.array([0, n], dtype=np.int64)
    iv = rng.integers(-50, 50, size=n).astype(S32)
    assert reduce(iv, off, "sum").tolist() == [int(iv.astype(np.int64).sum())]
    for dt in (S32, U32):
        x = iv.astype(dt)
        out, arg = reduce(x, off, "min")
        assert out.tolist() == [x.min()] and arg.tolist() == [int(np.argmin(x))]
        out, arg = reduce(x, off, "max")
        assert out.tolist() == [x.max()] and arg.tolist() == [int(np.argmax(x))]
    fv = rng.standard_normal(n).astype(F32)
    s = float(reduce(fv, off, "sum")[0])
    exact = math.fsum(fv.astype(np.float64))
    assert abs(s - exact) <= _f32_ulp(exact) + n * 2.0**-53 * float(np.abs(fv).sum())
    m = float(reduce(fv, off, "mean")[0])
    assert abs(m - exact / n) <= 2 * _f32_ulp(exact / n) + n * 2.0**-53 * float(np.abs(fv).sum()) / n


def pin_invariants(reduce):
    """graph-reduce README, 'Correctness': every arg gathers back to the
    reported value, lies in its segment, and no lower row of the segment
    holds an equal value; per-segment integer sums add up to the global sum
    mod 2^32; min <= mean <= max."""
    rng = np.random.default_rng(5)
    n, S = 3000, 200
    cuts = np.sort(rng.integers(0, n + 1, size=S - 1))
    off = np.concatenate([[0], cuts, [n]]).astype(np.int64)
    b, e = off[:-1], off[1:]
    fv = rng.integers(-20, 20, size=n).astype(F32)      # many ties
    for dt in (F32, S32, U32):
        v = fv.astype(dt) if dt is not U32 else fv.astype(S32).view(U32)
        for op in ("min", "max"):
            out, arg = reduce(v, off, op)
            for s in range(S):
                if e[s] == b[s]:
                    assert arg[s] == -1 and out[s] == 0
                    continue
                assert b[s] <= arg[s] < e[s]
                assert v[arg[s]] == out[s]
                seg = v[b[s]:e[s]]
                assert not np.any(seg[: arg[s] - b[s]] == out[s])
                assert (seg >= out[s]).all() if op == "min" else (seg <= out[s]).all()
    iv = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(U32)
    sums = reduce(iv, off, "sum").astype(np.uint64)
    assert int(sums.sum()) % 2**32 == int(iv.astype(np.uint64).sum()) % 2**32
    mn, _ = reduce(fv, off, "min")
    mx, _ = reduce(fv, off, "max")
    mean = reduce(fv, off, "mean")
    assert (mn <= mean).all() and (mean <= mx).all()


def pin_brute_force(reduce):
    """Tiny random inputs against the independent pure-Python restatement:
    integers and min / max exactly; float sums within one float32 ulp of the
    correctly rounded sum plus the double-accumulation bound."""
    rng = np.random.default_rng(13)
    for trial in range(40):
        n = int(rng.integers(0, 60))
        S = int(rng.integers(0, 12))
        F = int(rng.choice([1, 1, 2, 3]))
        cuts = np.sort(rng.integers(0, n + 1, size=max(S - 1, 0)))
        start = int(rng.integers(0, 3)) if n > 3 and S > 0 else 0
        cuts = np.clip(cuts, start, n)
        off = np.concatenate([[start], cuts, [n]])[: S + 1] if S > 0 else np.array([start])
        if S > 0:
            off[-1] = max(off[-1], off[-2]) if S > 1 else off[-1]
            off = np.maximum.accumulate(off)
        off = off.astype(np.int64 if trial % 2 else np.uint32)
        for kind, dt in (("u32", U32), ("s32", S32), ("f32", F32)):
            if kind == "f32":
                raw = rng.standard_normal((n, F)) * 10
                raw[rng.random((n, F)) < 0.2] = 1.5            # ties
                v = raw.astype(F32)
            else:
                v = rng.integers(-2**31, 2**31, size=(n, F)).astype(np.int64).astype(dt)
            arr = v if F > 1 else np.ascontiguousarray(v[:, 0])
            rows = v.tolist()
            ops = ("sum", "min", "max") + (("mean",) if kind == "f32" else ())
            for op in ops:
                got = reduce(arr, off, op)
                want, want_arg = brute.seg_reduce(rows, off.astype(np.int64).tolist(), op, kind, F)
                out = got[0] if isinstance(got, tuple) else got
                out = out.reshape(len(want), F) if len(want) else out.reshape(0, F)
                if op in ("min", "max"):
                    assert got[1].reshape(len(want), F).tolist() == want_arg, (trial, kind, op)
                if kind == "f32" and op in ("sum", "mean"):
                    for s in range(len(want)):
                        seg = v[off[s]:off[s + 1]].astype(np.float64)
                        for f in range(F):
                            bound = _f32_ulp(want[s][f]) + (len(seg) + 1) * 2.0**-53 * float(np.abs(seg[:, f]).sum())
                            if op == "mean" and len(seg):
                                bound = 2 * _f32_ulp(want[s][f]) + bound / len(seg)
                            assert abs(float(out[s, f]) - want[s][f]) <= bound, (trial, op, s, f)
                else:
                    assert out.tolist() == want, (trial, kind, op)


ALL_PINS = [
    pin_luma_worked_example, pin_luma_worked_example_derived, pin_rle_example,
    pin_empty_segments, pin_no_segments, pin_nonzero_first_offset,
    pin_closed_forms, pin_integer_wrap_and_order, pin_ties_lower_row,
    pin_signed_zero_ties, pin_row_tensor, pin_row_tensor_is_per_column,
    pin_single_segment_is_global_reduction, pin_invariants, pin_brute_force,
]
