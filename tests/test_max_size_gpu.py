"""Inputs past 2^31 elements on the GPU: the 64-bit index paths of the
scalar kernel, the row kernel, the scan, the offsets producers and the
scatter path (atomic and sorted).

At these sizes no CPU reference is run.  The values are ones with a few
planted entries, so every expected result has a closed form that holds at
any size (luma.gl GPUSegmentedReduction, "What is segmented reduction?"):
- a segment's sum is its length plus the planted deltas, modulo 2^32 for
  integers;
- min and max are 1 or a planted value, and the arg is the lowest row that
  holds it;
- an empty segment gives 0 and arg -1;
- the inclusive scan at row i is i - start + 1 plus the deltas planted at or
  before i.

The offsets put segment boundaries just below and above 2^31 rows. One
segment spans more than 2^31 rows.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

N = (1 << 31) + 3 * (1 << 20) + 5
OFFSETS = [0, 7, 1 << 20, (1 << 31) - 3, (1 << 31) + (1 << 19), (1 << 31) + (1 << 19), N - 1, N]
# row -> value; everything else is 1
PLANTED = {5: 0, (1 << 31) + 100: 7, (1 << 31) + 101: 7, (1 << 31) - 4: 9, N - 1: 42}


def _need_memory(nbytes):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes + (2 << 30):
        pytest.skip(f"needs {nbytes / 2**30:.1f} GiB of free device memory")


def _segment_expect(a, b, planted, op, modulo=None):
    """Closed form for a segment [a, b) of ones with `planted` entries."""
    if b <= a:
        return 0, -1
    inside = {r: v for r, v in planted.items() if a <= r < b}
    if op == "sum":
        s = (b - a) + sum(v - 1 for v in inside.values())
        return (s % modulo if modulo else s), None
    first_one = a
    while first_one in inside:
        first_one += 1
    cands = [(v, r) for r, v in inside.items()]
    if first_one < b:
        cands.append((1, first_one))
    if op == "min":
        v = min(c[0] for c in cands)
    else:
        v = max(c[0] for c in cands)
    return v, min(r for val, r in cands if val == v)


def _ones_with(dtype, planted):
    v = torch.ones(N, dtype=dtype, device="cuda")
    for r, x in planted.items():
        v[r] = x
    return v


def test_scalar_kernel_past_2_31_rows():
    import segmented_reduction_csr_gb300 as sr
    _need_memory(4 * N)
    off = torch.tensor(OFFSETS, dtype=torch.int64, device="cuda")
    segs = list(zip(OFFSETS[:-1], OFFSETS[1:]))
    v = _ones_with(torch.int32, PLANTED)
    for view in (torch.int32, torch.uint32):
        x = v.view(view)
        got = sr.seg_reduce(x, off, "sum").view(torch.int32).cpu().numpy().astype(np.int64) % (1 << 32)
        want = [_segment_expect(a, b, PLANTED, "sum", 1 << 32)[0] for a, b in segs]
        assert got.tolist() == want, (view, "sum")
        for op in ("min", "max"):
            o, arg = sr.seg_reduce(x, off, op)
            want = [_segment_expect(a, b, PLANTED, op) for a, b in segs]
            assert o.view(torch.int32).cpu().tolist() == [w[0] for w in want], (view, op)
            assert arg.cpu().tolist() == [w[1] for w in want], (view, op, "arg")
    del v, x
    torch.cuda.empty_cache()
    f = _ones_with(torch.float32, PLANTED)
    s = sr.seg_reduce(f, off, "sum").double().cpu().numpy()
    m = sr.seg_reduce(f, off, "mean").double().cpu().numpy()
    for k, (a, b) in enumerate(segs):
        exact = _segment_expect(a, b, PLANTED, "sum")[0]
        abs_sum = exact   # every value is non-negative
        assert abs(s[k] - exact) <= 1e-5 * abs_sum + 1e-6, (k, s[k], exact)
        if b > a:
            mean = np.float32(np.float32(exact) / np.float32(b - a))
            assert abs(m[k] - mean) <= 1e-5 * abs(mean) + 1e-6, (k, m[k], mean)
        else:
            assert m[k] == 0.0
    for op in ("min", "max"):
        o, arg = sr.seg_reduce(f, off, op)
        want = [_segment_expect(a, b, PLANTED, op) for a, b in segs]
        assert o.cpu().tolist() == [float(w[0]) for w in want], op
        assert arg.cpu().tolist() == [w[1] for w in want], (op, "arg")
    assert sr.device_status() == 0


def test_row_kernel_past_2_31_elements():
    import segmented_reduction_csr_gb300 as sr
    R, F = (1 << 25) + 3, 64          # R * F = 2^31 + 192 elements
    _need_memory(4 * R * F)
    roffs = [0, 5, 1 << 24, (1 << 25) + 1, (1 << 25) + 1, R]
    planted = {((1 << 25) - 1, 63): 9.0, (3, 0): -2.0, (R - 1, 17): 5.0}
    v = torch.ones((R, F), dtype=torch.float32, device="cuda")
    for (r, c), x in planted.items():
        v[r, c] = x
    off = torch.tensor(roffs, dtype=torch.int64, device="cuda")
    segs = list(zip(roffs[:-1], roffs[1:]))
    col_planted = [{r: x for (r, c), x in planted.items() if c == col} for col in range(F)]
    s = sr.seg_reduce(v, off, "sum").double().cpu().numpy()
    for k, (a, b) in enumerate(segs):
        for col in range(F):
            exact = _segment_expect(a, b, col_planted[col], "sum")[0]
            abs_sum = (b - a) + sum(abs(x) - 1 for r, x in col_planted[col].items() if a <= r < b)
            assert abs(s[k, col] - exact) <= 1e-5 * abs_sum + 1e-6, (k, col, s[k, col], exact)
    for op in ("min", "max"):
        o, arg = sr.seg_reduce(v, off, op)
        o, arg = o.cpu().numpy(), arg.cpu().numpy()
        for k, (a, b) in enumerate(segs):
            for col in range(F):
                val, row = _segment_expect(a, b, col_planted[col], op)
                assert o[k, col] == val and arg[k, col] == row, (op, k, col, o[k, col], arg[k, col], val, row)
    assert sr.device_status() == 0


def test_scan_past_2_31_rows():
    import segmented_reduction_csr_gb300 as sr
    _need_memory(8 * N)
    off = torch.tensor(OFFSETS, dtype=torch.int64, device="cuda")
    v = _ones_with(torch.int32, PLANTED).view(torch.uint32)
    out = sr.seg_scan(v, off, "sum")
    # sampled rows: every segment's ends, the rows around 2^31 and the
    # planted rows, and a seeded random sample
    rows = set()
    for a, b in zip(OFFSETS[:-1], OFFSETS[1:]):
        rows.update(r for r in (a, a + 1, b - 2, b - 1) if a <= r < b)
    for r in list(PLANTED) + [(1 << 31) - 1, 1 << 31, (1 << 31) + 1, N - 2]:
        rows.update({r - 1, r, r + 1})
    rng = np.random.default_rng(31)
    rows.update(int(x) for x in rng.integers(0, N, 2000))
    rows = sorted(r for r in rows if 0 <= r < N)
    idx = torch.tensor(rows, dtype=torch.int64, device="cuda")
    got = out.view(torch.int32)[idx].cpu().numpy().astype(np.int64) % (1 << 32)
    starts = np.array(OFFSETS[:-1])
    ends = np.array(OFFSETS[1:])
    for r, g in zip(rows, got.tolist()):
        s = int(np.nonzero((starts <= r) & (r < ends))[0][-1])
        a = OFFSETS[s]
        want = (r - a + 1) + sum(x - 1 for p, x in PLANTED.items() if a <= p <= r)
        assert g == want % (1 << 32), (r, g, want)
    assert sr.device_status() == 0


RUN_STARTS = [0, 5, 6, 1 << 20, (1 << 31) - 2, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, (1 << 31) + 77, N - 1]


def test_producers_past_2_31_elements():
    import segmented_reduction_csr_gb300 as sr
    _need_memory(4 * N + 4 * N + 4 * N + 8 * N)
    keys = torch.empty(N, dtype=torch.int32, device="cuda")
    bounds = RUN_STARTS + [N]
    for k, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        keys[a:b] = 3 * k + 1          # consecutive runs differ
    values, lengths, offsets = sr.rle(keys)
    assert values.cpu().tolist() == [3 * k + 1 for k in range(len(RUN_STARTS))]
    assert lengths.view(torch.int32).cpu().tolist() == [b - a for a, b in zip(bounds[:-1], bounds[1:])]
    assert offsets.cpu().tolist() == bounds
    del keys, values, lengths, offsets
    torch.cuda.empty_cache()
    flags = torch.zeros(N, dtype=torch.uint8, device="cuda")
    flags[torch.tensor(RUN_STARTS[1:], dtype=torch.int64, device="cuda")] = 1
    # index 0 is left unflagged: the offsets list the flagged indices only, then n
    got = sr.flags_to_offsets(flags).cpu().tolist()
    assert got == RUN_STARTS[1:] + [N]
    assert sr.device_status() == 0


def test_scatter_past_2_31_rows():
    import segmented_reduction_csr_gb300 as sr
    _need_memory(4 * N + 8 * N + 16 * N + 4 * N)
    SH = 21
    D = ((N - 1) >> SH) + 1
    src = torch.ones(N, dtype=torch.float32, device="cuda")
    planted = {3: -5.0, (1 << 31) + 100: 7.0, (1 << 31) + 101: 7.0, (1 << 31) - 9: 4.0}
    for r, x in planted.items():
        src[r] = x
    index = torch.arange(N, dtype=torch.int64, device="cuda") >> SH
    index[N - 1] = -1                  # goes nowhere
    dst = [{r: x for r, x in planted.items() if (r >> SH) == d} for d in range(D)]
    ranges = [(d << SH, min((d + 1) << SH, N - 1)) for d in range(D)]

    def expect(op):
        return [_segment_expect(a, b, dst[d], op) for d, (a, b) in enumerate(ranges)]

    for det in (False, True):
        s = sr.scatter(src, index, D, "sum", deterministic=det).double().cpu().numpy()
        assert s.tolist() == [float(e[0]) for e in expect("sum")], det
        torch.cuda.empty_cache()
    for op in ("max", "min"):
        o, arg = sr.scatter(src, index, D, op)
        want = expect(op)
        assert o.cpu().tolist() == [float(w[0]) for w in want], op
        assert arg.cpu().tolist() == [w[1] for w in want], (op, "arg")
    assert sr.device_status() == 0
