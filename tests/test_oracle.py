"""The CPU oracle against its pins (no GPU needed)."""
import numpy as np
import pytest

import oracle
from oracle import brute
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.seg_reduce)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_brute_force_pin(pin):
    """The pure-Python restatement satisfies the same pins (except the one
    that compares it with itself)."""
    if pin is oracle_pins.pin_brute_force:
        pytest.skip("compares brute force with the C oracle")

    def reduce(values, offsets, op):
        v = np.asarray(values)
        kind = {np.dtype(np.uint32): "u32", np.dtype(np.int32): "s32",
                np.dtype(np.float32): "f32"}[v.dtype]
        rows = (v.reshape(-1, 1) if v.ndim == 1 else v).tolist()
        if v.shape[0] == 0:
            rows = []
        f = 1 if v.ndim == 1 else v.shape[1]
        out, arg = brute.seg_reduce(rows, np.asarray(offsets).astype(np.int64).tolist(), op, kind, f)
        out = np.array(out, dtype=v.dtype).reshape(-1, f)
        arg = np.array(arg, dtype=np.int64).reshape(-1, f)
        if v.ndim == 1:
            out, arg = out[:, 0], arg[:, 0]
        return (out, arg) if op in ("min", "max") else out

    pin(reduce)


def test_oracle_rejects_bad_input():
    v = np.arange(5, dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.seg_reduce(v, np.array([0, 3, 2], dtype=np.int64), "sum")     # decreasing
    with pytest.raises(ValueError):
        oracle.seg_reduce(v, np.array([0, 6], dtype=np.int64), "sum")        # beyond N
    with pytest.raises(ValueError):
        oracle.seg_reduce(v.astype(np.int32), np.array([0, 5]), "mean")     # integer mean
    with pytest.raises(TypeError):
        oracle.seg_reduce(v.astype(np.float64), np.array([0, 5]), "sum")


def test_oracle_agrees_with_torch_segment_reduce():
    """graph-reduce README, 'Correctness', names torch.segment_reduce as its
    bitwise reference; on non-empty segments its CPU kernel is an
    independent check of values (float sums within rounding)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(17)
    lengths = rng.integers(1, 30, size=100)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    v = rng.standard_normal(int(off[-1])).astype(np.float32)
    for op, red in (("sum", "sum"), ("mean", "mean"), ("min", "min"), ("max", "max")):
        ref = torch.segment_reduce(torch.from_numpy(v), red,
                                   lengths=torch.from_numpy(lengths)).numpy()
        got = oracle.seg_reduce(v, off, op)
        got = got[0] if isinstance(got, tuple) else got
        if op in ("min", "max"):
            assert np.array_equal(got, ref)
        else:
            np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


def test_all_cores_build_equals_sequential_build():
    """The benchmark's all-cores CPU baseline times the same C loop built with
    OpenMP over (segment, column) pairs; every output must be bit for bit
    the sequential build's (each pair runs the same sequential inner loop)."""
    try:
        oracle.load_parallel_library()
    except Exception as e:   # no OpenMP in this gcc: the baseline reports one core
        pytest.skip(f"no OpenMP build: {e}")
    rng = np.random.default_rng(23)
    lengths = rng.integers(0, 60, size=5000)
    lengths[::11] = 0
    lengths[7] = 40_000
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    n = int(off[-1])
    for feat in (1, 5):
        shape = (n,) if feat == 1 else (n, feat)
        cases = {"f32": rng.standard_normal(shape).astype(np.float32),
                 "s32": rng.integers(-2**31, 2**31, size=shape).astype(np.int32)}
        cases["u32"] = cases["s32"].view(np.uint32)
        for kind, v in cases.items():
            for op in ("sum", "min", "max") + (("mean",) if kind == "f32" else ()):
                a = oracle.seg_reduce(v, off, op)
                b = oracle.seg_reduce_parallel(v, off, op)
                if isinstance(a, tuple):
                    assert np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32)), (feat, kind, op)
                    assert np.array_equal(a[1], b[1]), (feat, kind, op)
                else:
                    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (feat, kind, op)
    assert oracle.parallel_threads() >= 1
