"""libsegreduce without a GPU: it loads, exports every function include/*.h
declares, plans launches on the host, and rejects bad arguments before any
CUDA call."""
import ctypes
import glob
import os
import re

import pytest

import segmented_reduction_csr_gb300 as sr
from segmented_reduction_csr_gb300 import build as srbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    srbuild.build()
    return sr.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(seg_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_abi():
    names = _declared_functions()
    assert {"seg_reduce", "seg_reduce_strerror", "seg_reduce_device_status",
            "seg_reduce_plan", "seg_reduce_version"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"


def test_version_and_strerror(lib):
    assert lib.seg_reduce_version() >= 10000
    for code in range(6):
        assert lib.seg_reduce_strerror(code)
    assert lib.seg_reduce_strerror(99) == b"unknown status"


def _call(lib, values=8, dtype=2, F=1, n=10, offsets=8, odt=1, S=3, op=0, out=8, arg=None):
    return lib.seg_reduce(values, dtype, F, n, offsets, odt, S, op, out, arg, None)


def test_host_checks_reject_before_any_cuda_call(lib):
    # Fake (aligned, non-null) pointers: every case returns before touching CUDA.
    assert _call(lib, dtype=7) == 1                      # bad dtype
    assert _call(lib, odt=5) == 1                        # bad offsets dtype
    assert _call(lib, op=9) == 1                         # bad op
    assert _call(lib, F=0) == 1                          # F < 1
    assert _call(lib, n=-1) == 1                         # negative N
    assert _call(lib, S=-1) == 1                         # negative S
    assert _call(lib, dtype=0, op=3) == 2                # mean on uint32
    assert _call(lib, dtype=1, op=3) == 2                # mean on int32
    assert _call(lib, F=4096) == 2                       # F above the maximum
    assert _call(lib, op=0, arg=8) == 1                  # sum with an arg buffer
    assert _call(lib, op=3, arg=8) == 1                  # mean with an arg buffer
    assert _call(lib, S=0, offsets=None, out=None) == 0  # nothing to do: no launch
    assert _call(lib, offsets=None) == 1                 # null offsets
    assert _call(lib, out=None) == 1                     # null out
    assert _call(lib, values=None) == 1                  # null values with N > 0
    assert _call(lib, values=6) == 1                     # misaligned values
    assert _call(lib, offsets=12) == 1                   # misaligned int64 offsets
    assert _call(lib, out=2) == 1                        # misaligned out
    assert _call(lib, op=1, arg=4) == 1                  # misaligned arg


def test_producer_host_checks_reject_before_any_cuda_call(lib):
    # seg_rle(keys, n, values, lengths, offsets, count, stream)
    assert lib.seg_rle(None, 5, None, None, None, 64, None) == 1          # keys NULL, n > 0
    assert lib.seg_rle(64, -1, None, None, None, 64, None) == 1           # n < 0
    assert lib.seg_rle(64, 1 << 32, None, None, None, 64, None) == 1      # n > UINT32_MAX
    assert lib.seg_rle(64, 5, None, None, None, None, None) == 1          # count NULL
    assert lib.seg_rle(66, 5, None, None, None, 64, None) == 1            # keys misaligned
    assert lib.seg_rle(64, 5, 66, None, None, 64, None) == 1              # values misaligned
    assert lib.seg_rle(64, 5, None, 66, None, 64, None) == 1              # lengths misaligned
    assert lib.seg_rle(64, 5, None, None, 68, 64, None) == 1              # offsets misaligned
    assert lib.seg_rle(64, 5, None, None, None, 68, None) == 1            # count misaligned
    # seg_flags_to_offsets(flags, n, offsets, count, stream)
    assert lib.seg_flags_to_offsets(None, 5, 64, 64, None) == 1           # flags NULL, n > 0
    assert lib.seg_flags_to_offsets(64, -2, 64, 64, None) == 1            # n < 0
    assert lib.seg_flags_to_offsets(64, 5, None, 64, None) == 1           # offsets NULL
    assert lib.seg_flags_to_offsets(64, 5, 64, None, None) == 1           # count NULL
    assert lib.seg_flags_to_offsets(65, 5, 68, 64, None) == 1             # offsets misaligned
    assert lib.seg_flags_to_offsets(65, 5, 64, 60, None) == 1             # count misaligned


def test_sequential_host_checks_reject_before_any_cuda_call(lib):
    # seg_reduce_sequential(values, F, N, offsets, offsets_dtype, S, op, out, stream)
    seq = lib.seg_reduce_sequential
    assert seq(64, 1, 10, 64, 1, 0, 0, 64, None) == 0            # S == 0: nothing to do
    assert seq(64, 1, 10, 64, 1, 3, 1, 64, None) == 1            # min: not an input-order op
    assert seq(64, 1, 10, 64, 1, 3, 2, 64, None) == 1            # max
    assert seq(64, 1, 10, 64, 7, 3, 0, 64, None) == 1            # bad offsets dtype
    assert seq(64, 0, 10, 64, 1, 3, 0, 64, None) == 1            # F < 1
    assert seq(64, 4096, 10, 64, 1, 3, 0, 64, None) == 2         # F above SEG_MAX_FEATURES
    assert seq(64, 1, -1, 64, 1, 3, 0, 64, None) == 1            # N < 0
    assert seq(None, 1, 10, 64, 1, 3, 0, 64, None) == 1          # values NULL with N > 0
    assert seq(64, 1, 10, None, 1, 3, 0, 64, None) == 1          # offsets NULL
    assert seq(64, 1, 10, 64, 1, 3, 0, None, None) == 1          # out NULL
    assert seq(66, 1, 10, 64, 1, 3, 0, 64, None) == 1            # values misaligned
    assert seq(64, 1, 10, 68, 1, 3, 0, 64, None) == 1            # int64 offsets misaligned
    assert seq(64, 1, 10, 64, 1, 3, 3, 66, None) == 1            # out misaligned


def test_scatter_host_checks_reject_before_any_cuda_call(lib):
    # seg_scatter(src, dtype, F, N, index, dim_size, op, out, out_arg, stream)
    sc = lib.seg_scatter
    assert sc(64, 2, 1, 10, 64, 0, 0, 64, None, None) == 0          # dim_size 0: nothing to do
    assert sc(64, 7, 1, 10, 64, 5, 0, 64, None, None) == 1          # bad dtype
    assert sc(64, 2, 1, 10, 64, 5, 9, 64, None, None) == 1          # bad op
    assert sc(64, 2, 0, 10, 64, 5, 0, 64, None, None) == 1          # F < 1
    assert sc(64, 2, 4096, 10, 64, 5, 0, 64, None, None) == 2       # F too large
    assert sc(64, 0, 1, 10, 64, 5, 3, 64, None, None) == 2          # mean on uint32
    assert sc(64, 2, 1, 10, 64, 5, 0, 64, 64, None) == 1            # arg with sum
    assert sc(64, 2, 1, 1 << 32, 64, 5, 2, 64, None, None) == 2     # rows do not fit 32 bits
    assert sc(64, 2, 2048, (1 << 32) - 2, 64, 5, 0, 64, None, None) == 2   # N * F above 2^40: more than one launch
    assert sc(None, 2, 1, 10, 64, 5, 0, 64, None, None) == 1        # src NULL
    assert sc(64, 2, 1, 10, None, 5, 0, 64, None, None) == 1        # index NULL
    assert sc(64, 2, 1, 10, 64, 5, 0, None, None, None) == 1        # out NULL
    assert sc(64, 2, 1, 10, 68, 5, 0, 64, None, None) == 1          # index misaligned
    assert sc(64, 2, 1, 10, 64, 5, 2, 64, 68, None) == 1            # arg misaligned
    assert sc(64, 2, 1, -1, 64, 5, 0, 64, None, None) == 1          # N < 0


def test_sorted_scatter_host_checks_reject_before_any_cuda_call(lib):
    sc = lib.seg_scatter_sorted
    assert sc(64, 2, 1, 10, 64, 0, 0, 64, None, None) == 0          # dim_size 0: nothing to do
    assert sc(64, 7, 1, 10, 64, 5, 0, 64, None, None) == 1          # bad dtype
    assert sc(64, 2, 1, 10, 64, 5, 9, 64, None, None) == 1          # bad op
    assert sc(64, 0, 1, 10, 64, 5, 3, 64, None, None) == 2          # mean on uint32
    assert sc(64, 2, 1, 10, 64, 5, 0, 64, 64, None) == 1            # arg with sum
    assert sc(64, 2, 1, 1 << 32, 64, 5, 2, 64, None, None) == 2     # rows do not fit 32 bits
    assert sc(64, 2, 1, 10, 64, 1 << 32, 2, 64, None, None) == 2    # outputs do not fit 32 bits
    assert sc(None, 2, 1, 10, 64, 5, 0, 64, None, None) == 1        # src NULL
    assert sc(64, 2, 1, 10, 68, 5, 0, 64, None, None) == 1          # index misaligned


def test_scan_host_checks_reject_before_any_cuda_call(lib):
    # seg_scan(values, dtype, N, offsets, offsets_dtype, S, op, exclusive, out, stream)
    sc = lib.seg_scan
    assert sc(64, 2, 0, 64, 1, 3, 0, 0, 64, None) == 0             # N == 0: nothing to do
    assert sc(64, 7, 10, 64, 1, 3, 0, 0, 64, None) == 1            # bad dtype
    assert sc(64, 2, 10, 64, 5, 3, 0, 0, 64, None) == 1            # bad offsets dtype
    assert sc(64, 2, 10, 64, 1, 3, 3, 0, 64, None) == 1            # mean is not a scan op
    assert sc(64, 2, 10, 64, 1, 3, 2, 1, 64, None) == 2            # exclusive max
    assert sc(64, 2, 10, 64, 1, 3, 0, 2, 64, None) == 1            # exclusive not 0 / 1
    assert sc(64, 2, -1, 64, 1, 3, 0, 0, 64, None) == 1           # N < 0
    assert sc(64, 2, 10, 64, 1, -1, 0, 0, 64, None) == 1           # S < 0
    assert sc(None, 2, 10, 64, 1, 3, 0, 0, 64, None) == 1          # values NULL
    assert sc(64, 2, 10, None, 1, 3, 0, 0, 64, None) == 1          # offsets NULL
    assert sc(64, 2, 10, 64, 1, 3, 0, 0, None, None) == 1          # out NULL
    assert sc(66, 2, 10, 64, 1, 3, 0, 0, 64, None) == 1            # values misaligned
    assert sc(64, 2, 10, 68, 1, 3, 0, 0, 64, None) == 1            # int64 offsets misaligned


def test_plan_shapes(lib):
    p = sr.plan("f32", 1, 16_000_000, "i64", 1_000_000, "sum", sm_count=152)
    assert p["grid"] == 152 and p["slot_threads"] == 1 and p["vec"] == 1
    assert p["block"] == 512 and p["kernel_variant"] == 4          # the scalar kernel
    assert p["smem_bytes"] <= 227 * 1024
    assert p["workspace_bytes"] >= 152 * 16 * 8 + 2 * 152 * 16 * 16  # unit tickets + partials
    p = sr.plan("f32", 64, 1_000_000, "i64", 10_000, "max", values_addr=256, sm_count=152)
    assert p["vec"] == 2 and p["slot_threads"] == 32 and p["vecs_per_thread"] == 1
    assert p["grid"] == 152 and p["block"] == 256
    p = sr.plan("f32", 128, 1_000_000, "i64", 10_000, "sum", values_addr=256, sm_count=152)
    assert p["vec"] == 4 and p["vecs_per_thread"] == 1
    p = sr.plan("f32", 64, 1_000_000, "i64", 10_000, "max", values_addr=260, sm_count=152)
    assert p["vec"] == 1 and p["vecs_per_thread"] == 2        # misaligned rows: one column per lane
    p = sr.plan("f32", 2048, 1000, "i64", 10, "sum", values_addr=256, sm_count=152)
    assert p["vec"] == 4 and p["vecs_per_thread"] == 16
    p = sr.plan("f32", 130, 1000, "i64", 10, "sum", values_addr=256, sm_count=152)
    assert p["vec"] == 2 and p["vecs_per_thread"] == 3
    p = sr.plan("u32", 1, 100, "u32", 10, "min", sm_count=152)
    assert p["grid"] == 1                                # tiny input: one CTA
    for F in (2, 3, 5, 8, 64, 100, 128, 130, 1000, 1024, 2048):
        for addr in (256, 260):
            for op in ("sum", "max"):
                p = sr.plan("f32", F, 10_000_000, "i64", 100_000, op, values_addr=addr)
                assert p["smem_bytes"] <= 227 * 1024
                assert 32 * p["vec"] * p["vecs_per_thread"] >= F > 32 * p["vec"] * (p["vecs_per_thread"] - 1)
                assert addr % (4 * p["vec"]) == 0 and F % p["vec"] == 0
                units = p["grid"] * p["block"] // 32
                assert units >= p["vecs_per_thread"]
                per = 4 + (8 if op == "max" else 0)
                assert p["workspace_bytes"] >= 2 * units * 32 * p["vec"] * per


def test_plan_weighs_ends_by_op_and_routes_small_calls(lib):
    # rows kernel: an end weighs 2 rows for sums, 5 when min / max store rows,
    # so the same small problem gets more ranges (a larger grid) for max
    ps = sr.plan("f32", 64, 2000, "i64", 1000, "sum", values_addr=256, sm_count=152)
    pm = sr.plan("f32", 64, 2000, "i64", 1000, "max", values_addr=256, sm_count=152)
    assert ps["grid"] == 4 and pm["grid"] == 7            # ceil(ceil((2000 + w * 1000) / 128) / 8)
    # F = 1 up to 16,384 rows and 4,096 segments: the one-CTA small-input kernel
    small = sr.plan("f32", 1, 16_384, "i64", 4_096, "sum", sm_count=152)
    assert small["grid"] == 1 and small["block"] == 1024 and small["kernel_variant"] == 8
    for n, s in ((16_385, 4_096), (16_384, 4_097)):
        big = sr.plan("f32", 1, n, "i64", s, "sum", sm_count=152)
        assert big["kernel_variant"] == 4                  # the scalar kernel


def test_plan_rejects(lib):
    with pytest.raises(sr.SegReduceError):
        sr.plan("s32", 1, 10, "i64", 2, "mean")
    with pytest.raises(sr.SegReduceError):
        sr.plan("f32", 4096, 10, "i64", 2, "sum")
    with pytest.raises(sr.SegReduceError):
        sr.plan("f32", 1, 2**33, "u32", 2, "sum")       # uint32 offsets cannot address N


def test_python_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    v = torch.zeros(4)
    off = torch.tensor([0, 4])
    with pytest.raises(ValueError, match="CUDA"):
        sr.seg_reduce(v, off, "sum")
