"""Helpers for the GPU parity tests: move numpy arrays to the device, run the
CUDA path through the binding, run the oracle on the same inputs, compare.

Bar (from the benchmark spec of the method): integer results, min / max
values and args and empty segments bit-exact; float32 sums within
1e-5 * sum(|x|) + 1e-6 per output (means: that bound over the length plus
one rounding of the division)."""
from __future__ import annotations

import numpy as np

import oracle

TOL_REL = 1e-5
TOL_ABS = 1e-6


def torch_mod():
    import torch
    return torch


def to_dev(a: np.ndarray, device="cuda"):
    torch = torch_mod()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device).view(torch.uint32)
    return torch.from_numpy(a).to(device)


def to_host(t) -> np.ndarray:
    torch = torch_mod()
    if t.dtype == torch.uint32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def gpu_reduce(values: np.ndarray, offsets: np.ndarray, op: str, dvals=None, doffs=None):
    import segmented_reduction_csr_gb300 as sr
    dv = to_dev(values) if dvals is None else dvals
    do = to_dev(offsets) if doffs is None else doffs
    r = sr.seg_reduce(dv, do, op)
    if isinstance(r, tuple):
        return to_host(r[0]), to_host(r[1])
    return to_host(r), None


def abs_sums(values: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """sum(|x|) per segment (and column), in float64, from a running prefix
    built block by block (a few hundred MB at a time, whatever the input
    size).  Offsets must be nondecreasing."""
    feat = int(np.prod(values.shape[1:], dtype=np.int64))
    v2 = values.reshape(values.shape[0], feat)
    n = v2.shape[0]
    off = offsets.astype(np.int64)
    pre = np.empty((off.shape[0], feat), dtype=np.float64)   # prefix at each offset
    carry = np.zeros(feat, dtype=np.float64)
    block = max(1, (1 << 24) // feat)
    lo = 0
    for r0 in range(0, n, block):
        r1 = min(n, r0 + block)
        cs = np.empty((r1 - r0 + 1, feat), dtype=np.float64)
        cs[0] = carry
        np.cumsum(np.abs(v2[r0:r1].astype(np.float64)), axis=0, out=cs[1:])
        cs[1:] += carry
        hi = int(np.searchsorted(off, r1, side="left"))
        pre[lo:hi] = cs[off[lo:hi] - r0]
        lo = hi
        carry = cs[-1]
    pre[lo:] = carry
    r = pre[1:] - pre[:-1]
    return r.reshape((offsets.shape[0] - 1,) + values.shape[1:])


def assert_parity(values, offsets, op, got, got_arg, exp=None, exp_arg=None, where=""):
    if exp is None:
        r = oracle.seg_reduce(values, offsets, op)
        exp, exp_arg = r if isinstance(r, tuple) else (r, None)
    assert got.shape == exp.shape, (where, got.shape, exp.shape)
    if op in ("min", "max"):
        assert np.array_equal(got_arg, exp_arg), (where, _first_diff(got_arg, exp_arg))
    if values.dtype == np.float32 and op in ("sum", "mean"):
        off = offsets.astype(np.int64)
        tol = TOL_REL * abs_sums(values, offsets) + TOL_ABS
        if op == "mean":
            lens = np.maximum(np.diff(off), 1).astype(np.float64)
            lens = lens.reshape((-1,) + (1,) * (values.ndim - 1))
            tol = tol / lens + 2.0**-23 * np.abs(exp.astype(np.float64))
        err = np.abs(got.astype(np.float64) - exp.astype(np.float64))
        bad = err > tol
        assert not bad.any(), (where, op, int(bad.sum()), float(err.max()))
        empty = (np.diff(off) == 0)
        if empty.any():
            assert (got[empty] == 0).all(), (where, "empty segment not 0")
    else:
        gb = got.view(np.uint32)
        eb = exp.view(np.uint32)
        assert np.array_equal(gb, eb), (where, op, _first_diff(gb, eb))


def _first_diff(a, b):
    idx = np.argwhere(a != b)
    if idx.size == 0:
        return None
    i = tuple(idx[0])
    return {"index": i, "got": a[i].item(), "want": b[i].item(), "count": len(idx)}
