"""The allocation-free entry point (seg_reduce_noalloc) against the oracle and seg_reduce.

Collected last on purpose: it must pass both in a fresh process (where its
first call does the per-device set-up) and after every other test has used
the allocating entry point on the same device.  Each case runs the
allocating entry point once and the allocation-free one twice in a row,
into fresh outputs filled with a sentinel, and compares every result with
the independent CPU oracle at the parity bar of the other GPU tests, and
with the allocating entry point bit for bit (both launch the same kernel
with the same shape)."""
import zlib

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as H
import workloads as W

pytestmark = pytest.mark.gpu


def _case(kind, feat, lengths_spec, seed):
    rng = np.random.default_rng(seed)
    if lengths_spec == "mixed":
        lengths = rng.integers(0, 40, size=60_000)
        lengths[rng.integers(0, lengths.size, size=20)] = rng.integers(50_000, 400_000, size=20)
        lengths[::97] = 0
        if feat > 1:   # keep the row cases small
            lengths = lengths[:2000]
    else:   # few long segments: every one crosses many warp units
        lengths = rng.integers(200_000, 2_000_000, size=7)
        lengths[3] = 0
    off = W.offsets_from_lengths(lengths)
    n = int(off[-1])
    shape = (n,) if feat == 1 else (n, feat)
    if kind == "f32":
        vals = rng.standard_normal(shape).astype(np.float32)
    elif kind == "s32":
        vals = rng.integers(-2**31, 2**31, size=shape, dtype=np.int64).astype(np.int32)
    else:
        vals = rng.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32)
    return vals, off


CASES = [
    ("f32", 1, "mixed", "sum", np.int64),
    ("f32", 1, "long", "sum", np.int64),
    ("f32", 1, "mixed", "mean", np.uint32),
    ("u32", 1, "mixed", "max", np.int64),
    ("s32", 1, "long", "min", np.uint32),
    ("u32", 1, "long", "sum", np.int64),
    ("f32", 64, "mixed", "max", np.int64),
    ("f32", 130, "mixed", "mean", np.int64),
]


@pytest.mark.parametrize("kind,feat,spec,op,odt", CASES)
def test_noalloc_matches_seg_reduce(kind, feat, spec, op, odt):
    import torch
    import segmented_reduction_csr_gb300 as sr
    vals, off = _case(kind, feat, spec, seed=zlib.crc32(f"{kind}{feat}{spec}{op}".encode()))
    off = off.astype(odt)
    dv, do = H.to_dev(vals), H.to_dev(off)
    want = sr.seg_reduce(dv, do, op)
    want, want_arg = want if isinstance(want, tuple) else (want, None)
    want_h = H.to_host(want)
    want_arg_h = H.to_host(want_arg) if want_arg is not None else None
    r = oracle.seg_reduce(vals, off, op)
    oracle_out, oracle_arg = r if isinstance(r, tuple) else (r, None)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.empty_like(want)
        out.view(torch.int32).fill_(7)                  # sentinel bits
        arg = torch.full_like(want_arg, -7) if want_arg is not None else None
        sr.seg_reduce_noalloc(dv, do, op, out, arg, status_word=status)
        torch.cuda.synchronize()
        got = H.to_host(out)
        got_arg = H.to_host(arg) if arg is not None else None
        H.assert_parity(vals, off, op, got, got_arg, exp=oracle_out, exp_arg=oracle_arg,
                        where=f"noalloc call {call}")
        assert np.array_equal(got.view(np.uint32), want_h.view(np.uint32)), f"call {call}"
        if got_arg is not None:
            assert np.array_equal(got_arg, want_arg_h)
    assert int(status.item()) == 0


def test_noalloc_allocates_nothing():
    """After set-up, repeated calls leave the device's free memory unchanged."""
    import torch
    import segmented_reduction_csr_gb300 as sr
    vals, off = _case("f32", 1, "mixed", seed=5)
    dv, do = H.to_dev(vals), H.to_dev(off)
    out = torch.empty(off.size - 1, dtype=torch.float32, device="cuda")
    sr.seg_reduce_noalloc(dv, do, "sum", out)       # set-up (first call on the device)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        sr.seg_reduce_noalloc(dv, do, "sum", out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    want = sr.seg_reduce(dv, do, "sum")
    torch.cuda.synchronize()
    assert np.array_equal(H.to_host(out).view(np.uint32), H.to_host(want).view(np.uint32))


def test_noalloc_rejects_calls_beyond_its_scratch():
    """Wide rows with min / max on a large grid need more than the fixed
    array: a clear error, nothing launched (the output keeps its sentinel)."""
    import torch
    import segmented_reduction_csr_gb300 as sr
    feat = 2048
    n, s = 50_000, 100
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = sr.plan("f32", feat, n, "i64", s, "max", values_addr=256, sm_count=sms)["workspace_bytes"]
    assert need > sr.NOALLOC_SCRATCH_BYTES
    dv = torch.zeros((n, feat), dtype=torch.float32, device="cuda")
    do = torch.linspace(0, n, s + 1, device="cuda").to(torch.int64)
    out = torch.full((s, feat), 3.0, device="cuda")
    with pytest.raises(sr.SegReduceError) as ei:
        sr.seg_reduce_noalloc(dv, do, "max", out)
    assert ei.value.status == 6
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    # a narrow call on the same device still works afterwards
    small = torch.ones(1000, dtype=torch.float32, device="cuda")
    soff = torch.tensor([0, 10, 10, 1000], dtype=torch.int64, device="cuda")
    sout = torch.empty(3, dtype=torch.float32, device="cuda")
    sr.seg_reduce_noalloc(small, soff, "sum", sout)
    assert sout.cpu().tolist() == [10.0, 0.0, 990.0]


def test_noalloc_near_the_limit():
    """Row max with two columns a lane (F = 64) on a full grid: the partials
    then fill most of the fixed array.  Every output and arg against the
    oracle, and bitwise against seg_reduce, on two calls in a row."""
    import torch
    import segmented_reduction_csr_gb300 as sr
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(64)
    lengths = rng.integers(0, 12, size=40_000)
    lengths[rng.integers(0, lengths.size, size=8)] = rng.integers(5_000, 20_000, size=8)
    off = W.offsets_from_lengths(lengths)
    n = int(off[-1])
    vals = np.round(rng.standard_normal((n, 64)) * 3).astype(np.float32)   # many ties
    dv, do = H.to_dev(vals), H.to_dev(off)
    pl = sr.plan("f32", 64, n, "i64", off.size - 1, "max", values_addr=dv.data_ptr(), sm_count=sms)
    assert pl["vec"] == 2 and pl["grid"] == sms
    assert 0.5 * sr.NOALLOC_SCRATCH_BYTES < pl["workspace_bytes"] <= sr.NOALLOC_SCRATCH_BYTES
    want, want_arg = sr.seg_reduce(dv, do, "max")
    exp, exp_arg = oracle.seg_reduce(vals, off, "max")
    for call in range(2):
        out = torch.full_like(want, 7.0)
        arg = torch.full_like(want_arg, -7)
        sr.seg_reduce_noalloc(dv, do, "max", out, arg)
        torch.cuda.synchronize()
        H.assert_parity(vals, off, "max", H.to_host(out), H.to_host(arg), exp=exp, exp_arg=exp_arg,
                        where=f"near limit, call {call}")
        assert torch.equal(out.view(torch.int32), want.view(torch.int32)) and torch.equal(arg, want_arg)


def test_noalloc_four_column_rows_follow_the_plan():
    """Row min / max that load four columns a lane (F % 4 == 0, F > 64,
    16-byte aligned rows; here F = 96) need 24 KiB of partials per CTA: a
    small grid fits and matches the oracle, a large one is refused before
    anything is launched."""
    import torch
    import segmented_reduction_csr_gb300 as sr
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(96)
    # small: a few thousand rows, grid well under the limit
    lengths = rng.integers(0, 30, size=200)
    off = W.offsets_from_lengths(lengths)
    n = int(off[-1])
    vals = rng.standard_normal((n, 96)).astype(np.float32)
    dv, do = H.to_dev(vals), H.to_dev(off)
    pl = sr.plan("f32", 96, n, "i64", off.size - 1, "min", values_addr=dv.data_ptr(), sm_count=sms)
    assert pl["vec"] == 4 and pl["workspace_bytes"] <= sr.NOALLOC_SCRATCH_BYTES
    out = torch.empty((off.size - 1, 96), device="cuda")
    arg = torch.empty((off.size - 1, 96), dtype=torch.int64, device="cuda")
    sr.seg_reduce_noalloc(dv, do, "min", out, arg)
    torch.cuda.synchronize()
    H.assert_parity(vals, off, "min", H.to_host(out), H.to_host(arg), where="F=96 small grid")
    # large: 200,000 rows of 96 columns on a full grid
    n2 = 200_000
    big = torch.zeros((n2, 96), dtype=torch.float32, device="cuda")
    boff = torch.linspace(0, n2, 1001, device="cuda").to(torch.int64)
    pl = sr.plan("f32", 96, n2, "i64", 1000, "max", values_addr=big.data_ptr(), sm_count=sms)
    assert pl["workspace_bytes"] > sr.NOALLOC_SCRATCH_BYTES
    bout = torch.full((1000, 96), 3.0, device="cuda")
    with pytest.raises(sr.SegReduceError) as ei:
        sr.seg_reduce_noalloc(big, boff, "max", bout)
    assert ei.value.status == 6
    torch.cuda.synchronize()
    assert bool((bout == 3.0).all())
