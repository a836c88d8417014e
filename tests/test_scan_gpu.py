"""GPU parity of the segmented scan against the CPU oracle, through the
library's C ABI.  Integer sums, min and max and the zeros of rows in no
segment are bit-exact; float32 sums are within 1e-5 * sum(|x| over the row's
prefix) + 1e-6 (the row's own rows only, as for the reduction's bound)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_helpers import TOL_ABS, TOL_REL, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sr():
    import segmented_reduction_csr_gb300 as m
    m.load_library()
    return m


def _values(rng, kind, n):
    if kind == "f32":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "s32":
        return rng.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32)
    return rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)


def _prefix_abs(v, off, exclusive):
    """sum(|x|) over each row's prefix within its segment (0 outside)."""
    a = np.abs(v.astype(np.float64))
    cs = np.concatenate([[0.0], np.cumsum(a)])
    off = off.astype(np.int64)
    out = np.zeros(v.shape[0])
    lengths = np.diff(off)
    seg_start = np.repeat(off[:-1], lengths)
    rows = np.arange(off[0], off[-1])
    end = rows if exclusive else rows + 1
    out[rows] = cs[end] - cs[seg_start]
    return out


def _check(sr, v, off, op, exclusive=False, dv=None, where=""):
    exp = oracle.seg_scan(v, off, op, exclusive)
    got = to_host(sr.seg_scan(to_dev(v) if dv is None else dv, to_dev(off), op, exclusive))
    if v.dtype == np.float32 and op == "sum":
        err = np.abs(got.astype(np.float64) - exp.astype(np.float64))
        tol = TOL_REL * _prefix_abs(v, off, exclusive) + TOL_ABS
        bad = np.flatnonzero(err > tol)
        assert bad.size == 0, f"{where}: {bad.size} rows off, first {bad[:5]}"
        outside = np.ones(v.shape[0], bool)
        outside[int(off[0]):int(off[-1])] = False
        assert not np.any(got[outside]), where
    else:
        bad = np.flatnonzero(got.view(np.uint32) != exp.view(np.uint32))
        assert bad.size == 0, f"{where}: {bad.size} rows differ, first {bad[:5]}"


SIZES = [1, 15, 16, 17, 4095, 4096, 4097, 3 * 4096 + 5, 100_003, 1_000_003]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind", ["u32", "s32", "f32"])
def test_random(sr, n, kind):
    rng = np.random.default_rng(n * 7 + len(kind))
    v = _values(rng, kind, n)
    segs = max(1, n // 20)
    off = W.random_offsets(rng, n, segs, empty_frac=0.15, start=n // 10, stop=n - n // 10)
    for op, excl in (("sum", False), ("sum", True), ("min", False), ("max", False)):
        _check(sr, v, off, op, excl, where=f"{kind} n={n} {op}{' excl' if excl else ''}")


@pytest.mark.parametrize("kind", ["u32", "f32"])
def test_one_segment_over_every_cta(sr, kind):
    rng = np.random.default_rng(3)
    n = 5_000_001
    v = _values(rng, kind, n) if kind != "f32" else rng.random(n).astype(np.float32)   # all positive
    off = np.array([0, n], np.int64)
    for op, excl in (("sum", False), ("sum", True), ("max", False)):
        _check(sr, v, off, op, excl, where=f"one segment {kind} {op}")


def test_long_and_short_segments(sr):
    rng = np.random.default_rng(5)
    lengths = np.array([1, 0, 300_000, 2, 70_000, 0, 0, 5, 1_000_000, 17, 4096, 4097] * 4)
    rng.shuffle(lengths)
    off = W.offsets_from_lengths(lengths)
    n = int(off[-1])
    v = rng.standard_normal(n).astype(np.float32)
    for op, excl in (("sum", False), ("sum", True), ("min", False), ("max", False)):
        _check(sr, v, off, op, excl, where=f"mixed {op}")


def test_no_segments_gives_zeros(sr):
    v = np.arange(1, 1001, dtype=np.int32)
    for off in (np.array([0], np.int64), np.array([500], np.int64), np.array([300, 300, 300], np.int64)):
        _check(sr, v, off, "sum", where=f"empty {off}")


def test_uint32_offsets_tiny_workload(sr):
    w = W.make("tiny")
    for kind in ("f32", "u32"):
        for op, excl in (("sum", False), ("sum", True), ("min", False), ("max", False)):
            _check(sr, w.values[kind], w.offsets, op, excl, where=f"tiny {kind} {op}")


def test_misaligned_values(sr):
    rng = np.random.default_rng(6)
    v = rng.standard_normal(200_001).astype(np.float32)
    base = to_dev(np.concatenate([np.zeros(1, np.float32), v]))
    dv = base[1:]
    assert dv.data_ptr() % 16 != 0
    off = W.random_offsets(rng, 200_001, 3000)
    _check(sr, v, off, "sum", dv=dv, where="misaligned")
    _check(sr, v, off, "max", dv=dv, where="misaligned max")


@pytest.mark.parametrize("name", ["bulk", "skewed"])
def test_full_workloads(sr, name):
    w = W.make(name)
    cases = [("s32", "sum", False), ("u32", "max", False), ("f32", "sum", False), ("f32", "min", False)] \
        if name == "bulk" else [("f32", "sum", False), ("f32", "sum", True), ("f32", "max", False)]
    for kind, op, excl in cases:
        _check(sr, w.values[kind], w.offsets, op, excl, where=f"{name} {kind} {op}")


def test_repeated_calls_identical(sr):
    import torch
    w = W.make("bulk")
    dv, do = to_dev(w.values["f32"]), to_dev(w.offsets)
    first = sr.seg_scan(dv, do, "sum").clone()
    for _ in range(3):
        assert torch.equal(sr.seg_scan(dv, do, "sum").view(torch.int32), first.view(torch.int32))
