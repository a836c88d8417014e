"""CUDA path vs the CPU oracle, element by element (needs a GB300).

Integers, min / max (values and args) and empty segments must match bit for
bit; float32 sums / means within 1e-5 * sum(|x|) + 1e-6 per output; float
results must be bitwise identical across repeated runs.
"""
import json
import os
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_helpers import assert_parity, gpu_reduce, to_dev, to_host

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DT = {"u32": np.uint32, "s32": np.int32, "f32": np.float32}


def _values(rng, n, kind, feat=1, ties=False):
    shape = (n,) if feat == 1 else (n, feat)
    if kind == "f32":
        v = rng.standard_normal(shape).astype(np.float32)
        if ties:
            v = np.round(v * 4).astype(np.float32)
        return v
    lo, hi = (-(1 << 20), 1 << 20) if not ties else (-8, 8)
    v = rng.integers(lo, hi, size=shape, endpoint=True).astype(np.int64)
    return v.astype(np.int32).view(np.uint32) if kind == "u32" else v.astype(np.int32)


def _check(values, offsets, op, where=""):
    got, arg = gpu_reduce(values, offsets, op)
    assert_parity(values, offsets, op, got, arg, where=where)


def _ops(kind):
    return ("sum", "min", "max", "mean") if kind == "f32" else ("sum", "min", "max")


# ---------------------------------------------------------------------------

def test_pages_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "luma_segmented_reduction_example.json")))
    for kind, dt in DT.items():
        for odt in (np.uint32, np.int64):
            v = np.array(g["values"], dtype=dt)
            off = np.array(g["offsets"], dtype=odt)
            for op in ("sum", "min", "max"):
                got, _ = gpu_reduce(v, off, op)
                assert got.tolist() == g["expected"][op], (kind, op)
    r = json.load(open(os.path.join(GOLDEN, "luma_run_length_example.json")))
    v = np.array(r["input"], dtype=np.int32)
    off = np.array(r["offsets"], dtype=np.int64)
    out, arg = gpu_reduce(v, off, "max")
    assert out.tolist() == r["run_values"] and arg.tolist() == r["offsets"][:-1]


@pytest.mark.parametrize("kind", ["f32", "u32", "s32"])
@pytest.mark.parametrize("shape", ["short", "empties", "long", "mixed", "few"])
def test_scalar_random(kind, shape):
    rng = np.random.default_rng(zlib.crc32(f"{kind}-{shape}".encode()))
    if shape == "short":
        lengths = rng.geometric(1 / 16, size=40_000)
    elif shape == "empties":
        lengths = rng.integers(0, 6, size=60_000) * (rng.random(60_000) < 0.5)
    elif shape == "long":
        lengths = rng.integers(100_000, 700_000, size=6)
    elif shape == "mixed":
        lengths = rng.zipf(1.6, size=30_000).clip(max=400_000)
        lengths[rng.random(lengths.size) < 0.2] = 0
    else:
        lengths = np.array([0, 1, 0, 0, 3_000_000, 0, 2, 1_500_000, 0])
    off = W.offsets_from_lengths(lengths)
    v = _values(rng, int(off[-1]), kind, ties=(shape == "mixed"))
    for op in _ops(kind):
        _check(v, off, op, where=(kind, shape, op))


@pytest.mark.parametrize("feat", [2, 3, 4, 5, 8, 16, 64, 100, 128, 130, 256, 512, 1024, 1030, 2048])
def test_rows_f32(feat):
    rng = np.random.default_rng(feat)
    n_target = max(2000, 6_000_000 // feat)
    lengths = rng.geometric(1 / 12, size=max(10, n_target // 12))
    lengths[rng.random(lengths.size) < 0.1] = 0
    lengths[len(lengths) // 2] = 3 * n_target // 4 if feat >= 64 else lengths[len(lengths) // 2]
    off = W.offsets_from_lengths(lengths)
    v = _values(rng, int(off[-1]), "f32", feat=feat, ties=(feat % 2 == 1))
    for op in ("sum", "mean", "min", "max"):
        _check(v, off, op, where=(feat, op))


@pytest.mark.parametrize("kind", ["u32", "s32"])
@pytest.mark.parametrize("feat", [3, 4, 64, 128])
def test_rows_int(kind, feat):
    rng = np.random.default_rng(7 * feat)
    lengths = rng.integers(0, 40, size=20_000 // feat + 50)
    off = W.offsets_from_lengths(lengths)
    v = _values(rng, int(off[-1]), kind, feat=feat, ties=True)
    for op in ("sum", "min", "max"):
        _check(v, off, op, where=(kind, feat, op))


@pytest.mark.parametrize("feat", [1, 4, 64])
def test_misaligned_values_base(feat):
    """values starting 4 bytes past a 16-byte boundary: plain-load head bytes
    and the scalar-column path."""
    import segmented_reduction_csr_gb300 as sr
    rng = np.random.default_rng(99 + feat)
    lengths = rng.integers(0, 30, size=5000)
    off = W.offsets_from_lengths(lengths)
    n = int(off[-1])
    flat = rng.standard_normal(n * feat + 1).astype(np.float32)
    dflat = to_dev(flat)
    dv = dflat[1:].view(n, feat) if feat > 1 else dflat[1:]
    assert dv.data_ptr() % 16 == 4
    v = flat[1:].reshape(n, feat) if feat > 1 else flat[1:]
    for op in ("sum", "max"):
        r = sr.seg_reduce(dv, to_dev(off), op)
        got, arg = (to_host(r[0]), to_host(r[1])) if isinstance(r, tuple) else (to_host(r), None)
        assert_parity(v, off, op, got, arg, where=(feat, op))


def test_nonzero_start_and_unreduced_tail():
    rng = np.random.default_rng(5)
    n = 500_000
    v = rng.standard_normal(n).astype(np.float32)
    off = np.sort(rng.integers(1000, n - 1000, size=2001)).astype(np.int64)
    for op in ("sum", "min", "max", "mean"):
        _check(v, off, op, where=op)
    vi = rng.integers(-100, 100, size=(n // 50, 8)).astype(np.int32)
    off2 = np.array([3, 3, 10, 400, 9000, 9001], dtype=np.int64)
    for op in ("sum", "min", "max"):
        _check(vi, off2, op, where=("rows", op))


def test_edge_sizes():
    rng = np.random.default_rng(6)
    v = rng.standard_normal(100_000).astype(np.float32)
    cases = {
        "no_rows": (np.zeros(0, np.float32), np.zeros(7, np.int64)),
        "all_empty": (v, np.full(5000, 777, np.int64)),
        "global": (v, np.array([0, v.size], np.int64)),
        "one_row": (v[:1].copy(), np.array([0, 1], np.int64)),
        "single_row_segments": (v[:9000].copy(), np.arange(9001, dtype=np.int64)),
    }
    for T in (8191, 8192, 8193, 16384, 24575):   # around the scalar tile size
        cases[f"len{T}"] = (v, np.array([0, T, 2 * T, 2 * T + 1, 4 * T], np.int64))
    for name, (vals, off) in cases.items():
        for op in ("sum", "min", "max", "mean"):
            _check(vals, off, op, where=(name, op))


def test_integer_extremes_and_signed_zero():
    off = np.array([0, 3, 6, 8], np.int64)
    u = np.array([0xFFFFFFFF, 0xFFFFFFFF, 1, 0, 0, 0, 0x80000000, 0x80000000], np.uint32)
    for op in ("sum", "min", "max"):
        _check(u, off, op, where=("u32", op))
        _check(u.view(np.int32), off, op, where=("s32", op))
    z = np.array([0.0, -0.0, 0.0, -0.0, -0.0, 0.0, 1.0, 1.0], np.float32)
    for op in ("min", "max"):
        _check(z, off, op, where=("zero", op))


def test_uint32_offsets():
    rng = np.random.default_rng(8)
    lengths = rng.integers(0, 50, size=50_000)
    off = W.offsets_from_lengths(lengths, np.uint32)
    v = _values(rng, int(off[-1]), "u32")
    for op in ("sum", "min", "max"):
        _check(v, off, op, where=op)


@pytest.mark.parametrize("feat", [1, 64, 100])
def test_shared_memory_search_matches_probe_search(feat):
    """Offsets arrays up to 96 KB are searched in shared memory, larger ones
    by probe rounds (the scalar kernel and the staged row kernel; F = 100
    takes the register-ring shape, which always probes).  With 20,000
    segments, uint32 offsets (80 KB) take the first search and int64 offsets
    (160 KB) the second.  For valid offsets both find the same partition, so
    the results match bit for bit -- float sums included -- and both match
    the oracle."""
    rng = np.random.default_rng(20 + feat)
    lengths = rng.integers(0, 2 * 48 // feat + 30, size=20_000)
    lengths[rng.integers(0, lengths.size, 40)] = 0
    off64 = W.offsets_from_lengths(lengths, np.int64)
    off32 = off64.astype(np.uint32)
    for kind in ("f32", "u32"):
        v = _values(rng, int(off64[-1]), kind, feat)
        dv = to_dev(v)
        d64, d32 = to_dev(off64), to_dev(off32)
        for op in _ops(kind):
            g64, a64 = gpu_reduce(v, off64, op, dvals=dv, doffs=d64)
            g32, a32 = gpu_reduce(v, off32, op, dvals=dv, doffs=d32)
            assert np.array_equal(g64.view(np.uint32), g32.view(np.uint32)), (feat, kind, op)
            if a64 is not None:
                assert np.array_equal(a64, a32), (feat, kind, op, "arg")
            assert_parity(v, off64, op, g64, a64, where=(feat, kind, op))


@pytest.mark.parametrize("S", [12_287, 12_288])
def test_shared_memory_search_threshold(S):
    """int64 offsets of 12,287 segments (96 KB with the end) are searched in
    shared memory, 12,288 by probe rounds: both sides of the boundary."""
    rng = np.random.default_rng(S)
    lengths = rng.integers(0, 40, size=S)
    off = W.offsets_from_lengths(lengths, np.int64)
    for feat in (1, 64):
        v = _values(rng, int(off[-1]), "f32", feat)
        for op in ("sum", "max"):
            _check(v, off, op, where=(S, feat, op))


def test_float_sums_are_bitwise_reproducible():
    import segmented_reduction_csr_gb300 as sr
    rng = np.random.default_rng(9)
    lengths = np.concatenate([rng.geometric(1 / 20, 20_000), [2_500_000, 0, 1_200_000]])
    rng.shuffle(lengths)
    off = W.offsets_from_lengths(lengths)
    v = rng.standard_normal(int(off[-1])).astype(np.float32)
    dv, do = to_dev(v), to_dev(off)
    first = to_host(sr.seg_reduce(dv, do, "sum"))
    for _ in range(9):
        again = to_host(sr.seg_reduce(dv, do, "sum"))
        assert np.array_equal(first.view(np.uint32), again.view(np.uint32))
    rows = rng.standard_normal((200_000, 64)).astype(np.float32)
    roff = W.offsets_from_lengths(np.array([150_000, 3, 0, 49_997]))
    dr, dro = to_dev(rows), to_dev(roff)
    first = to_host(sr.seg_reduce(dr, dro, "mean"))
    for _ in range(9):
        assert np.array_equal(first.view(np.uint32), to_host(sr.seg_reduce(dr, dro, "mean")).view(np.uint32))


def test_two_streams_and_preallocated_outputs():
    import segmented_reduction_csr_gb300 as sr
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    lengths = rng.integers(0, 100, size=30_000)
    off = W.offsets_from_lengths(lengths)
    v = rng.standard_normal(int(off[-1])).astype(np.float32)
    dv, do = to_dev(v), to_dev(off)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1 = torch.empty(off.size - 1, device="cuda")
    o2 = torch.empty(off.size - 1, device="cuda")
    a2 = torch.empty(off.size - 1, device="cuda", dtype=torch.int64)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        sr.seg_reduce(dv, do, "sum", out=o1)
    with torch.cuda.stream(s2):
        sr.seg_reduce(dv, do, "max", out=o2, out_arg=a2)
    torch.cuda.synchronize()
    assert_parity(v, off, "sum", to_host(o1), None)
    e, ea = oracle.seg_reduce(v, off, "max")
    assert_parity(v, off, "max", to_host(o2), to_host(a2), e, ea)


def test_malformed_offsets_do_not_fault():
    """The luma contract leaves offsets unvalidated; the kernels clamp them, so a
    decreasing or out-of-range offsets array gives unspecified values but
    touches no memory outside the arguments and leaves no error behind."""
    import segmented_reduction_csr_gb300 as sr
    torch = pytest.importorskip("torch")
    v = to_dev(np.arange(1000, dtype=np.float32))
    for off in ([0, 500, 200, 1000], [0, 5000, 10, 20], [900, 100], [0, 10**9, 2 * 10**9]):
        o = to_dev(np.array(off, np.int64))
        for op in ("sum", "max"):
            sr.seg_reduce(v, o, op)
    torch.cuda.synchronize()
    assert sr.device_status() == 0
    # and a following well-formed call is still exact
    _check(np.arange(1000, dtype=np.float32), np.array([0, 10, 1000], np.int64), "sum")


# ---------------------------------------------------------------------------
# The five synthetic workloads at full size, in the configuration the
# benchmark times: every output and arg against the oracle, and every case
# run ten times with results bitwise equal to the first run (float sums
# included: the combine order is fixed).

def _workload_cases(name, w):
    extra = (("f32", "mean"),) if name in ("skewed", "bulk", "large") else ()
    return w.cases + extra


@pytest.mark.parametrize("name", ["tiny", "bulk", "mp", "skewed", "large"])
def test_workload_full(name):
    import segmented_reduction_csr_gb300 as sr
    torch = pytest.importorskip("torch")
    w = W.make(name)
    dvals = {k: to_dev(a) for k, a in w.values.items()}
    doffs = to_dev(w.offsets)
    for kind, op in _workload_cases(name, w):
        got, arg = gpu_reduce(w.values[kind], w.offsets, op, dvals=dvals[kind], doffs=doffs)
        assert_parity(w.values[kind], w.offsets, op, got, arg, where=(name, kind, op))
        # ten runs, bitwise identical (compared on the device)
        first = sr.seg_reduce(dvals[kind], doffs, op)
        first, first_arg = first if isinstance(first, tuple) else (first, None)
        for run in range(9):
            again = sr.seg_reduce(dvals[kind], doffs, op)
            again, again_arg = again if isinstance(again, tuple) else (again, None)
            assert torch.equal(again.view(torch.int32), first.view(torch.int32)), (name, kind, op, run)
            if first_arg is not None:
                assert torch.equal(again_arg, first_arg), (name, kind, op, run, "arg")
        # and the first of those is the one compared with the oracle above
        assert np.array_equal(to_host(first).view(np.uint32), got.view(np.uint32)), (name, kind, op)


def test_calls_with_changing_grids_share_scratch():
    """Calls on one stream share the library's scratch; a small-grid call
    followed by larger-grid calls (and back) must not disturb the cross-CTA
    tickets of the later calls."""
    rng = np.random.default_rng(12)
    layouts = []
    for nseg, mean_len in ((300, 40), (40_000, 16), (2_000, 400), (120_000, 20), (10, 200_000)):
        lengths = rng.geometric(1 / mean_len, size=nseg)
        off = W.offsets_from_lengths(lengths)
        layouts.append((off, rng.standard_normal(int(off[-1])).astype(np.float32)))
    for _ in range(3):
        for off, v in layouts:
            for op in ("sum", "max"):
                _check(v, off, op, where=(off.size, op))


@pytest.mark.parametrize("kind", ["f32", "u32", "s32"])
def test_small_input_shape(kind):
    """F == 1 inputs of at most 16,384 rows and 4,096 segments take the
    one-CTA shape: short segments by a thread, longer ones by a warp.  Both
    sides of both limits, segments of 32 and 33 rows (the thread / warp
    split), long segments with many ties, empties, a non-zero first offset,
    uint32 offsets; every output and arg against the oracle."""
    import segmented_reduction_csr_gb300 as sr
    rng = np.random.default_rng(zlib.crc32(f"small-{kind}".encode()))
    layouts = []
    for n, s in ((16_384, 4_096), (16_385, 4_096), (16_384, 4_097), (3_000, 200), (1, 1)):
        cuts = np.sort(rng.integers(0, n + 1, size=s - 1))
        off = np.concatenate([[0], cuts, [n]]).astype(np.int64)
        layouts.append((n, off))
    lengths = np.array([32, 33, 0, 31, 1, 5_000, 64, 0, 2_000, 97])
    off = W.offsets_from_lengths(lengths)
    layouts.append((int(off[-1]), off))
    layouts.append((9_000, np.array([17, 17, 40, 2_000, 2_001, 8_000], np.int64)))   # o0 > 0, tail unreduced
    for n, off in layouts:
        v = _values(rng, n, kind, ties=True)
        small = sr.plan(kind, 1, n, "i64", off.size - 1, "sum")["kernel_variant"] == 8
        assert small == (n <= 16_384 and off.size - 1 <= 4_096)
        for odt in (np.int64, np.uint32):
            for op in _ops(kind):
                _check(v, off.astype(odt), op, where=(kind, n, off.size, odt.__name__, op))
