"""GPU parity of the unsorted scatter path (graph-reduce README, "API" and
"Method") against the CPU oracle, through the library's C ABI.  Integer sums,
max / min values and args and empty outputs are bit-exact; float32 sums are
within 1e-5 * sum(|x|) + 1e-6 per output (atomics land in varying order), and
means within that bound over the count plus one rounding."""
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


def _values(rng, kind, shape):
    if kind == "f32":
        return rng.standard_normal(shape).astype(np.float32)
    if kind == "s32":
        return rng.integers(-2**31, 2**31, size=shape, dtype=np.int64).astype(np.int32)
    return rng.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32)


def _abs_sums(v, idx, dim):
    v2 = np.abs(v.astype(np.float64)).reshape(v.shape[0], -1)
    acc = np.zeros((dim, v2.shape[1]))
    ok = (idx >= 0) & (idx < dim)
    np.add.at(acc, idx[ok], v2[ok])
    return acc.reshape((dim,) + v.shape[1:])


def _check(sr, v, idx, dim, op, dv=None, where=""):
    exp = oracle.scatter(v, idx, dim, op)
    got = sr.scatter(to_dev(v) if dv is None else dv, to_dev(idx), dim, op)
    if op in ("min", "max"):
        (eo, ea), (go, ga) = exp, (to_host(got[0]), to_host(got[1]))
        assert np.array_equal(go.view(np.uint32), eo.view(np.uint32)), f"{where} {op} values"
        assert np.array_equal(ga, ea), f"{where} {op} args"
        return
    got = to_host(got)
    if v.dtype != np.float32:
        assert np.array_equal(got, exp), f"{where} {op}"
        return
    tol = TOL_REL * _abs_sums(v, idx, dim) + TOL_ABS
    if op == "mean":
        cnt = np.bincount(idx[(idx >= 0) & (idx < dim)], minlength=dim).astype(np.float64)
        cnt = cnt.reshape((dim,) + (1,) * (v.ndim - 1))
        tol = tol / np.maximum(cnt, 1) + np.abs(exp.astype(np.float64)) * 2.0 ** -23
    err = np.abs(got.astype(np.float64) - exp.astype(np.float64))
    assert np.all(err <= tol), f"{where} {op}: worst {np.max(err - tol)}"


@pytest.mark.parametrize("kind", ["u32", "s32", "f32"])
@pytest.mark.parametrize("feat", [1, 3, 4, 16, 64, 130])
def test_random(sr, kind, feat):
    rng = np.random.default_rng(1000 * ("u32", "s32", "f32").index(kind) + feat)
    n, dim = 30_011, 997
    v = _values(rng, kind, (n,) if feat == 1 else (n, feat))
    idx = rng.integers(0, dim, size=n).astype(np.int64)
    for op in ("sum", "min", "max") + (("mean",) if kind == "f32" else ()):
        _check(sr, v, idx, dim, op, where=f"{kind} F={feat}")


@pytest.mark.parametrize("dim", [1, 3])
def test_heavy_contention(sr, dim):
    """Every row into one to three outputs: ties among equal values must go
    to the lowest row."""
    rng = np.random.default_rng(dim)
    v = rng.integers(0, 4, size=(200_000, 8)).astype(np.float32)     # many ties
    idx = rng.integers(0, dim, size=200_000).astype(np.int64)
    for op in ("sum", "min", "max", "mean"):
        _check(sr, v, idx, dim, op, where=f"dim={dim}")


def test_out_of_range_and_empty_outputs(sr):
    rng = np.random.default_rng(9)
    v = rng.standard_normal((5000, 5)).astype(np.float32)
    idx = rng.integers(-50, 300, size=5000).astype(np.int64)      # negatives and >= dim skipped
    idx[idx % 7 == 0] = 10**12
    for op in ("sum", "min", "max", "mean"):
        _check(sr, v, idx, 400, op, where="out of range")


def test_signed_zeros_tie(sr):
    v = np.array([0.0, -0.0, -0.0, 0.0, -1.0, -0.0], np.float32)
    idx = np.array([0, 0, 1, 1, 2, 2], np.int64)
    for op in ("max", "min"):
        _check(sr, v, idx, 3, op, where="zeros")


def test_misaligned_src_takes_scalar_reductions(sr):
    rng = np.random.default_rng(4)
    v = rng.standard_normal((4001, 8)).astype(np.float32)
    base = to_dev(np.concatenate([np.zeros(1, np.float32), v.ravel()]))
    dv = base[1:].view(4001, 8)
    assert dv.data_ptr() % 16 != 0
    idx = rng.integers(0, 50, size=4001).astype(np.int64)
    _check(sr, v, idx, 50, "sum", dv=dv, where="misaligned")


def test_no_rows(sr):
    import torch
    out = sr.scatter(torch.zeros((0, 4), dtype=torch.float32, device="cuda"),
                     torch.zeros(0, dtype=torch.int64, device="cuda"), 6, "max")
    assert to_host(out[0]).tolist() == [[0.0] * 4] * 6 and to_host(out[1]).tolist() == [[-1] * 4] * 6


def test_message_passing_shape_full_size(sr):
    """graph-reduce README "Measured" row: 1,000,000 rows x 64 float32 into
    10,000 outputs, destinations uniform and unsorted."""
    v, idx, dim = W.scatter_input("mp")
    dv = to_dev(v)
    for op in ("sum", "max", "mean"):
        _check(sr, v, idx, dim, op, dv=dv, where="mp")


def test_integer_and_extreme_results_repeat_exactly(sr):
    import torch
    rng = np.random.default_rng(12)
    v = rng.integers(-1000, 1000, size=(300_000, 16)).astype(np.int32)
    idx = to_dev(rng.integers(0, 123, size=300_000).astype(np.int64))
    dv = to_dev(v)
    for op in ("sum", "max"):
        first = sr.scatter(dv, idx, 123, op)
        first = first[0] if isinstance(first, tuple) else first
        for _ in range(3):
            again = sr.scatter(dv, idx, 123, op)
            again = again[0] if isinstance(again, tuple) else again
            assert torch.equal(first, again), op
