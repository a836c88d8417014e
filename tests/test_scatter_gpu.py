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
    for op in ("sum", "min", "max"):   # min / max: one column an item
        _check(sr, v, idx, 50, op, dv=dv, where="misaligned")


@pytest.mark.parametrize("order", ["rising", "falling"])
@pytest.mark.parametrize("kind", ["u32", "s32", "f32"])
def test_extremes_along_monotone_rows(sr, order, kind):
    """max / min skip an element's atomic when its output already holds a
    better value.  Values that rise along the rows make every element of a
    max improve on its output (each reaches its atomic) and nearly every
    element of a min lose; falling values the reverse.  Runs of equal values
    (ties, settled by the atomic: the lowest row wins) and the type's extreme
    values are mixed in.  Both must give the one-atomic-per-element result."""
    rng = np.random.default_rng(("rising", "falling").index(order) * 10 + ("u32", "s32", "f32").index(kind))
    n, feat, dim = 60_000, 8, 37
    v = np.sort(_values(rng, kind, (n, feat)), axis=0)
    m = v[1::7].shape[0]
    v[0::7][:m] = v[1::7]   # equal neighbours (the order stays monotone)
    if kind == "s32":
        v[:50] = np.iinfo(np.int32).min
        v[-50:] = np.iinfo(np.int32).max
    elif kind == "u32":
        v[:50] = 0
        v[-50:] = np.iinfo(np.uint32).max
    if order == "falling":
        v = v[::-1].copy()
    idx = rng.integers(0, dim, size=n).astype(np.int64)
    dv = to_dev(v)
    for op in ("max", "min"):
        _check(sr, v, idx, dim, op, dv=dv, where=f"{order} {kind}")


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


# ---- the deterministic scatter (sort by destination, then the segmented path) ----------

def _sorted_reference(sr, v, idx, dim, op):
    """seg_reduce over all rows stably sorted on the host by destination (an
    index outside [0, dim) taken as dim, so those rows sort last and lie in
    no segment), args mapped back to the original rows.  All N rows stay in
    the array: the reduction's fixed float order depends on its row count."""
    ok = (idx >= 0) & (idx < dim)
    key = np.where(ok, idx, dim)
    perm = np.argsort(key, kind="stable")
    off = np.concatenate([[0], np.cumsum(np.bincount(idx[ok], minlength=dim))]).astype(np.int64)
    r = sr.seg_reduce(to_dev(np.ascontiguousarray(v[perm])), to_dev(off), op)
    if isinstance(r, tuple):
        o, a = to_host(r[0]), to_host(r[1])
        return o, np.where(a >= 0, perm[np.maximum(a, 0)], -1)
    return to_host(r), None


@pytest.mark.parametrize("dim", [1, 300, 70_000])
@pytest.mark.parametrize("feat", [1, 8, 64])
def test_sorted_scatter_equals_segmented_path_over_sorted_rows(sr, dim, feat):
    """Bit for bit: the device sort is stable and the reduction is the
    segmented path's (1, 2 and 3 radix passes)."""
    rng = np.random.default_rng(dim + feat)
    n = 50_003
    v = rng.standard_normal((n,) if feat == 1 else (n, feat)).astype(np.float32)
    idx = rng.integers(-3, dim + 3, size=n).astype(np.int64)
    for op in ("sum", "mean", "max", "min"):
        got = sr.scatter(to_dev(v), to_dev(idx), dim, op, deterministic=True)
        exp, exp_arg = _sorted_reference(sr, v, idx, dim, op)
        if isinstance(got, tuple):
            assert np.array_equal(to_host(got[0]).view(np.uint32), exp.view(np.uint32)), op
            assert np.array_equal(to_host(got[1]), exp_arg), op
        else:
            assert np.array_equal(to_host(got).view(np.uint32), exp.view(np.uint32)), op


@pytest.mark.parametrize("kind", ["u32", "s32", "f32"])
def test_sorted_scatter_against_the_oracle(sr, kind):
    rng = np.random.default_rng(7 + len(kind))
    v = _values(rng, kind, (40_000, 5))
    idx = rng.integers(0, 777, size=40_000).astype(np.int64)
    for op in ("sum", "max", "min") + (("mean",) if kind == "f32" else ()):
        exp = oracle.scatter(v, idx, 777, op)
        got = sr.scatter(to_dev(v), to_dev(idx), 777, op, deterministic=True)
        if op in ("max", "min"):
            assert np.array_equal(to_host(got[0]).view(np.uint32), exp[0].view(np.uint32)), op
            assert np.array_equal(to_host(got[1]), exp[1]), op
        elif kind != "f32":
            assert np.array_equal(to_host(got), exp), op
        else:
            err = np.abs(to_host(got).astype(np.float64) - exp.astype(np.float64))
            tol = TOL_REL * _abs_sums(v, idx, 777) + TOL_ABS
            if op == "mean":
                cnt = np.bincount(idx, minlength=777).astype(np.float64)[:, None]
                tol = tol / np.maximum(cnt, 1) + np.abs(exp.astype(np.float64)) * 2.0 ** -23
            assert np.all(err <= tol), op


def test_sorted_scatter_is_bitwise_reproducible_and_handles_no_rows(sr):
    import torch
    v, idx, dim = W.scatter_input("mp")
    dv, di = to_dev(v), to_dev(idx)
    first = sr.scatter(dv, di, dim, "sum", deterministic=True).clone()
    for _ in range(3):
        again = sr.scatter(dv, di, dim, "sum", deterministic=True)
        assert torch.equal(again.view(torch.int32), first.view(torch.int32))
    exp, _ = _sorted_reference(sr, v, idx, dim, "sum")
    assert np.array_equal(to_host(first).view(np.uint32), exp.view(np.uint32))
    o, a = sr.scatter(torch.zeros((0, 4), dtype=torch.float32, device="cuda"),
                      torch.zeros(0, dtype=torch.int64, device="cuda"), 5, "max", deterministic=True)
    assert not to_host(o).any() and (to_host(a) == -1).all()
