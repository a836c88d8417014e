"""GPU parity of the input-order float32 mode (graph-reduce README,
"Correctness": a fixed summation order) against the CPU oracle, through the
library's C ABI.  Both sides add in input order with float32 rounding, so the
bar is bitwise equality of every output."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sr():
    import segmented_reduction_csr_gb300 as m
    m.load_library()
    return m


def _check(sr, values, offsets, op, where=""):
    exp = oracle.seg_reduce_sequential(values, offsets, op)
    got = to_host(sr.seg_reduce_sequential(to_dev(values), to_dev(offsets), op))
    assert got.shape == exp.shape, where
    bad = np.flatnonzero(got.view(np.uint32).ravel() != exp.view(np.uint32).ravel())
    assert bad.size == 0, f"{where}: {bad.size} outputs differ, first at {bad[:5]}"


def _wide(rng, shape):
    # magnitudes over 11 decades: the order of the additions shows in the bits
    return (rng.standard_normal(shape) * 10.0 ** rng.integers(-3, 8, size=shape)).astype(np.float32)


@pytest.mark.parametrize("feat", [1, 3, 32, 33, 64, 100])
@pytest.mark.parametrize("op", ["sum", "mean"])
def test_random_shapes(sr, feat, op):
    rng = np.random.default_rng(100 + feat)
    n = 20_011
    v = _wide(rng, (n,) if feat == 1 else (n, feat))
    off = W.random_offsets(rng, n, 700, empty_frac=0.2)
    _check(sr, v, off, op, f"F={feat}")


@pytest.mark.parametrize("feat", [1, 64])
def test_long_and_short_segments_mixed(sr, feat):
    """Lengths around and far above the long-segment threshold (512 rows),
    several long segments in one warp, next to short and empty ones."""
    rng = np.random.default_rng(77 + feat)
    lengths = np.array([0, 3, 511, 512, 513, 1000, 0, 7, 33, 100_000, 1, 2048, 40_000, 5, 600, 601] * 5)
    rng.shuffle(lengths)
    off = W.offsets_from_lengths(lengths)
    n = int(off[-1])
    v = _wide(rng, (n,) if feat == 1 else (n, feat))
    for op in ("sum", "mean"):
        _check(sr, v, off, op, f"mixed F={feat} {op}")


def test_rows_outside_the_offsets_are_ignored(sr):
    rng = np.random.default_rng(5)
    v = _wide(rng, (5000, 7))
    off = W.random_offsets(rng, 5000, 60, start=123, stop=4321)
    _check(sr, v, off, "sum")
    _check(sr, v, off, "mean")


def test_uint32_offsets_and_order_sensitive_rows(sr):
    v = np.array([1e8, -1e8, 1, 1e8, 1, -1e8, 1, 1, -1e8, 1e8, -0.0], np.float32)
    off = np.array([0, 3, 7, 10, 11, 11], np.uint32)
    got = to_host(sr.seg_reduce_sequential(to_dev(v), to_dev(off), "sum"))
    assert list(got.view(np.uint32)) == list(np.array([1.0, 1.0, 0.0, 0.0, 0.0], np.float32).view(np.uint32))
    _check(sr, v, off, "mean")


def test_no_segments(sr):
    import torch
    v = torch.zeros(10, dtype=torch.float32, device="cuda")
    out = sr.seg_reduce_sequential(v, torch.zeros(1, dtype=torch.int64, device="cuda"))
    assert out.numel() == 0


def test_tiny_workload(sr):
    w = W.make("tiny")
    for op in ("sum", "mean"):
        _check(sr, w.values["f32"], w.offsets, op, "tiny")


@pytest.mark.parametrize("name,ops", [("bulk", ("sum", "mean")), ("mp", ("sum", "mean")),
                                      ("skewed", ("sum",)), ("large", ("sum",))])
def test_full_workloads(sr, name, ops):
    w = W.make(name)
    for op in ops:
        _check(sr, w.values["f32"], w.offsets, op, f"{name} {op}")


def test_repeated_calls_identical(sr):
    import torch
    w = W.make("mp")
    dv, do = to_dev(w.values["f32"]), to_dev(w.offsets)
    first = sr.seg_reduce_sequential(dv, do, "sum").clone()
    for _ in range(5):
        assert torch.equal(sr.seg_reduce_sequential(dv, do, "sum").view(torch.int32), first.view(torch.int32))


@pytest.mark.parametrize("feat", [1, 3, 64, 128])
def test_matches_torch_segment_reduce(sr, feat):
    """graph-reduce README, "Correctness": bitwise equal to
    torch.segment_reduce.  Rows [N, F] are compared with torch's CUDA
    segment_reduce; [N] with torch's CPU one (torch's CUDA [N] path adds in
    another order).  Empty segments are left out of the mean (torch's is
    NaN, this mode's is 0)."""
    import torch
    rng = np.random.default_rng(40 + feat)
    n = 60_000
    shape = (n,) if feat == 1 else (n, feat)
    v = _wide(rng, shape)
    off = W.random_offsets(rng, n, 900, empty_frac=0.1)
    nonempty = np.diff(off) > 0
    for op in ("sum", "mean"):
        got = to_host(sr.seg_reduce_sequential(to_dev(v), to_dev(off), op))
        if feat == 1:
            ref = torch.segment_reduce(torch.from_numpy(v), op, offsets=torch.from_numpy(off),
                                       axis=0, unsafe=True).numpy()
        else:
            ref = torch.segment_reduce(to_dev(v), op, offsets=to_dev(off), axis=0, unsafe=True).cpu().numpy()
        assert np.array_equal(got[nonempty].view(np.uint32), ref[nonempty].view(np.uint32)), op


def test_binding_rejects(sr):
    import torch
    v = torch.zeros(8, dtype=torch.int32, device="cuda")
    off = torch.tensor([0, 8], dtype=torch.int64, device="cuda")
    with pytest.raises(TypeError):
        sr.seg_reduce_sequential(v, off)
    with pytest.raises(ValueError):
        sr.seg_reduce_sequential(v.float(), off, "max")
    with pytest.raises(ValueError):
        sr.seg_reduce_sequential(v.float().cpu(), off.cpu())
