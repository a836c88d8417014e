"""segmented_reduction_csr_gb300 -- segmented reduction over offset-delimited
(CSR indptr) segments on NVIDIA GB300 (sm_103a).

A thin ctypes binding of ``libsegreduce.so`` (C ABI in ``include/seg_reduce.h``).
Every step of the reduction runs in the library's CUDA kernels; this module
only checks shapes, allocates outputs with torch and passes raw pointers and
the current CUDA stream.  There is no CPU fallback: if the library is
missing or no GPU is present, the calls raise.

Semantics (GPUSegmentedReduction "Contract"; graph-reduce README "API"):
segment ``s`` reduces rows ``[indptr[s], indptr[s+1])`` of ``src`` (``[N]`` or
``[N, F]``, over dimension 0); ``sum`` / ``min`` / ``max`` for uint32, int32
and float32, ``mean`` for float32; ``min`` / ``max`` also return the absolute
source row (int64; ties to the lower row; -1 for an empty segment); empty
segments give 0.

Beside the reduction (``seg_reduce``, ``segment_*_csr``, ``seg_reduce_noalloc``):

* ``seg_reduce_sequential``: float32 sum / mean added in input order
  (bitwise equal to an in-order float32 loop, as torch.segment_reduce);
* ``scatter`` / ``scatter_{sum,add,mean,max,min}``: the unsorted path, one
  atomic per element (graph-reduce README "API"; max / min skip the atomic
  of an element its output already beats);
* ``seg_scan`` / ``segment_cumsum_csr``: segmented inclusive / exclusive scan;
* ``seg_rle`` / ``rle`` / ``unique`` and ``seg_flags_to_offsets`` /
  ``flags_to_offsets``: producers of offsets (GPURunLengthEncode, GPUUnique,
  GPUSegmentedLayout).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "seg_reduce", "segment_sum_csr", "segment_mean_csr", "segment_min_csr",
    "segment_max_csr", "plan", "device_status", "library_path", "load_library",
    "SegReduceError", "seg_reduce_noalloc", "NOALLOC_SCRATCH_BYTES",
    "seg_rle", "rle", "unique", "seg_flags_to_offsets", "flags_to_offsets",
    "seg_reduce_sequential", "scatter", "scatter_sum", "scatter_add", "scatter_mean",
    "scatter_max", "scatter_min", "seg_scan", "segment_cumsum_csr",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libsegreduce.so")

# Codes of include/seg_reduce.h
SEG_U32, SEG_S32, SEG_F32 = 0, 1, 2
SEG_OFF_U32, SEG_OFF_I64 = 0, 1
OPS = {"sum": 0, "min": 1, "max": 2, "mean": 3}
STATUS = {0: "SEG_OK", 1: "SEG_ERR_INVALID_ARGUMENT", 2: "SEG_ERR_UNSUPPORTED",
          3: "SEG_ERR_OUT_OF_MEMORY", 4: "SEG_ERR_CUDA", 5: "SEG_ERR_DEVICE_TIMEOUT",
          6: "SEG_ERR_SCRATCH_LIMIT"}
EXPORTED = ("seg_reduce", "seg_reduce_strerror", "seg_reduce_device_status",
            "seg_reduce_plan", "seg_reduce_version", "seg_reduce_noalloc", "seg_rle",
            "seg_flags_to_offsets", "seg_reduce_sequential", "seg_scatter", "seg_scatter_sorted", "seg_scan",
            "seg_selftest_wait_timeout")
NOALLOC_SCRATCH_BYTES = 2 << 20   # SEG_NOALLOC_SCRATCH_BYTES


class SegReduceError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_strerror(status)})")


class _Plan(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("slot_threads", ctypes.c_int32), ("items_per_slot", ctypes.c_int32),
                ("vec", ctypes.c_int32), ("vecs_per_thread", ctypes.c_int32),
                ("max_ends", ctypes.c_int32), ("kernel_variant", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load libsegreduce.so (raises OSError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"{p} is missing: build it with "
                          "`python -m segmented_reduction_csr_gb300.build`")
        lib = ctypes.CDLL(p)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.seg_reduce.restype = ctypes.c_int
        lib.seg_reduce.argtypes = [vp, ctypes.c_int, i64, i64, vp, ctypes.c_int, i64,
                                   ctypes.c_int, vp, vp, vp]
        lib.seg_reduce_strerror.restype = ctypes.c_char_p
        lib.seg_reduce_strerror.argtypes = [ctypes.c_int]
        lib.seg_reduce_device_status.restype = ctypes.c_int
        lib.seg_reduce_device_status.argtypes = [vp]
        lib.seg_reduce_plan.restype = ctypes.c_int
        lib.seg_reduce_plan.argtypes = [ctypes.c_int, i64, i64, ctypes.c_int, i64, ctypes.c_int,
                                        ctypes.c_uint64, i32, ctypes.POINTER(_Plan)]
        lib.seg_reduce_version.restype = i32
        lib.seg_reduce_version.argtypes = []
        lib.seg_reduce_noalloc.restype = ctypes.c_int
        lib.seg_reduce_noalloc.argtypes = [vp, ctypes.c_int, i64, i64, vp, ctypes.c_int, i64,
                                           ctypes.c_int, vp, vp, vp, vp]
        lib.seg_rle.restype = ctypes.c_int
        lib.seg_rle.argtypes = [vp, i64, vp, vp, vp, vp, vp]
        lib.seg_flags_to_offsets.restype = ctypes.c_int
        lib.seg_flags_to_offsets.argtypes = [vp, i64, vp, vp, vp]
        lib.seg_selftest_wait_timeout.restype = ctypes.c_int
        lib.seg_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        lib.seg_scan.restype = ctypes.c_int
        lib.seg_scan.argtypes = [vp, ctypes.c_int, i64, vp, ctypes.c_int, i64, ctypes.c_int, i32, vp, vp]
        lib.seg_scatter_sorted.restype = ctypes.c_int
        lib.seg_scatter_sorted.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, ctypes.c_int, vp, vp, vp]
        lib.seg_scatter.restype = ctypes.c_int
        lib.seg_scatter.argtypes = [vp, ctypes.c_int, i64, i64, vp, i64, ctypes.c_int, vp, vp, vp]
        lib.seg_reduce_sequential.restype = ctypes.c_int
        lib.seg_reduce_sequential.argtypes = [vp, i64, i64, vp, ctypes.c_int, i64, ctypes.c_int, vp, vp]
        if path is None:
            _lib = lib
        return lib


def _strerror(status: int) -> str:
    try:
        return load_library().seg_reduce_strerror(status).decode()
    except OSError:
        return "library not loaded"


def plan(dtype: str, feat: int, num_values: int, offsets_dtype: str, num_segments: int,
         op: str, values_addr: int = 0, sm_count: int = 152) -> dict:
    """The launch the library would make (host-only; no GPU needed)."""
    pl = _Plan()
    rc = load_library().seg_reduce_plan(
        {"u32": SEG_U32, "s32": SEG_S32, "f32": SEG_F32}[dtype], feat, num_values,
        {"u32": SEG_OFF_U32, "i64": SEG_OFF_I64}[offsets_dtype], num_segments, OPS[op],
        values_addr, sm_count, ctypes.byref(pl))
    if rc != 0:
        raise SegReduceError(rc, "seg_reduce_plan")
    return {f: getattr(pl, f) for f, _ in _Plan._fields_}


def _torch():
    import torch
    return torch


def _value_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return SEG_F32
    if t.dtype == torch.int32:
        return SEG_S32
    if t.dtype == getattr(torch, "uint32", None):
        return SEG_U32
    raise TypeError(f"values must be float32, int32 or uint32, not {t.dtype}")


def _offset_code(t):
    torch = _torch()
    if t.dtype == torch.int64:
        return SEG_OFF_I64
    if t.dtype == getattr(torch, "uint32", None):
        return SEG_OFF_U32
    raise TypeError(f"offsets must be int64 or uint32, not {t.dtype}")


def seg_reduce(values, offsets, op: str = "sum", out=None, out_arg=None, with_arg: bool = True,
               stream=None):
    """Reduce ``values`` ([N] or [N, F], CUDA) over the segments that ``offsets``
    ([S+1], CUDA, int64 or uint32) delimits.

    Returns ``out`` for sum / mean, ``(out, arg)`` for min / max when
    ``with_arg`` (arg int64, -1 for empty segments).  ``out`` / ``out_arg`` may
    be passed preallocated.  Work is enqueued on ``stream`` (default: the
    current stream of the values' device) and is not synchronised.
    """
    torch = _torch()
    if op not in OPS:
        raise ValueError(f"op must be one of {sorted(OPS)}")
    if not values.is_cuda or not offsets.is_cuda:
        raise ValueError("values and offsets must be CUDA tensors (there is no CPU path)")
    if values.device != offsets.device:
        raise ValueError("values and offsets must be on the same device")
    if values.dim() not in (1, 2) or offsets.dim() != 1 or offsets.numel() < 1:
        raise ValueError("values must be [N] or [N, F] and offsets [S+1]")
    if not values.is_contiguous() or not offsets.is_contiguous():
        raise ValueError("values and offsets must be contiguous")
    lib = load_library()
    n = values.shape[0]
    feat = 1 if values.dim() == 1 else values.shape[1]
    s = offsets.numel() - 1
    oshape = (s,) if values.dim() == 1 else (s, feat)
    if out is None:
        out = torch.empty(oshape, dtype=values.dtype, device=values.device)
    elif tuple(out.shape) != oshape or out.dtype != values.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {values.dtype} tensor of shape {oshape}")
    want_arg = op in ("min", "max") and (with_arg or out_arg is not None)
    if want_arg and out_arg is None:
        out_arg = torch.empty(oshape, dtype=torch.int64, device=values.device)
    if out_arg is not None and (tuple(out_arg.shape) != oshape or out_arg.dtype != torch.int64
                                or not out_arg.is_contiguous()):
        raise ValueError(f"out_arg must be a contiguous int64 tensor of shape {oshape}")
    if stream is None:
        stream = torch.cuda.current_stream(values.device)
    with torch.cuda.device(values.device):
        rc = lib.seg_reduce(values.data_ptr() if n else None, _value_code(values), feat, n,
                            offsets.data_ptr(), _offset_code(offsets), s, OPS[op],
                            out.data_ptr() if s else None,
                            out_arg.data_ptr() if (want_arg and s) else None,
                            ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_reduce")
    return (out, out_arg) if want_arg else out


def seg_reduce_noalloc(values, offsets, op: str, out, out_arg=None, status_word=None,
                       stream=None):
    """``seg_reduce`` through the library's allocation-free entry point.

    For callers that may not allocate device memory when they reduce: neither
    the library (its scratch is a fixed static device array of
    ``NOALLOC_SCRATCH_BYTES``) nor this wrapper allocates anything, so ``out``
    (and ``out_arg`` to receive min / max rows) must be passed preallocated.
    ``status_word`` is an optional caller-owned int32 / uint32 CUDA tensor of
    one element that a timed-out device wait ORs a code into.  Calls whose
    kernels could overlap in time (other streams, other threads) race on the
    one array per device.  Raises ``SegReduceError`` with
    ``SEG_ERR_SCRATCH_LIMIT`` when the call needs more scratch than the array
    holds (large grids with wide rows).  Returns what ``seg_reduce`` returns.
    """
    torch = _torch()
    if op not in OPS:
        raise ValueError(f"op must be one of {sorted(OPS)}")
    if not values.is_cuda or not offsets.is_cuda:
        raise ValueError("values and offsets must be CUDA tensors (there is no CPU path)")
    if values.device != offsets.device:
        raise ValueError("values and offsets must be on the same device")
    if values.dim() not in (1, 2) or offsets.dim() != 1 or offsets.numel() < 1:
        raise ValueError("values must be [N] or [N, F] and offsets [S+1]")
    if not values.is_contiguous() or not offsets.is_contiguous():
        raise ValueError("values and offsets must be contiguous")
    n = values.shape[0]
    feat = 1 if values.dim() == 1 else values.shape[1]
    s = offsets.numel() - 1
    oshape = (s,) if values.dim() == 1 else (s, feat)
    if (out is None or tuple(out.shape) != oshape or out.dtype != values.dtype
            or not out.is_contiguous() or out.device != values.device):
        raise ValueError(f"out must be a preallocated contiguous {values.dtype} CUDA tensor "
                         f"of shape {oshape}")
    if out_arg is not None and (op not in ("min", "max") or tuple(out_arg.shape) != oshape
                                or out_arg.dtype != torch.int64 or not out_arg.is_contiguous()
                                or out_arg.device != values.device):
        raise ValueError(f"out_arg must be a contiguous int64 CUDA tensor of shape {oshape}, "
                         "for min / max only")
    if status_word is not None and (status_word.numel() != 1 or status_word.element_size() != 4
                                    or status_word.device != values.device):
        raise ValueError("status_word must be a one-element 32-bit CUDA tensor")
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(values.device)
    with torch.cuda.device(values.device):
        rc = lib.seg_reduce_noalloc(
            values.data_ptr() if n else None, _value_code(values), feat, n,
            offsets.data_ptr(), _offset_code(offsets), s, OPS[op],
            out.data_ptr() if s else None,
            out_arg.data_ptr() if (out_arg is not None and s) else None,
            status_word.data_ptr() if status_word is not None else None,
            ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_reduce_noalloc")
    return (out, out_arg) if out_arg is not None else out


def segment_sum_csr(src, indptr):
    """Per-segment sum of ``src`` rows (graph-reduce README, ``segment_sum_csr``)."""
    return seg_reduce(src, indptr, "sum")


def segment_mean_csr(src, indptr):
    """Per-segment mean; an empty segment gives 0."""
    return seg_reduce(src, indptr, "mean")


def segment_max_csr(src, indptr):
    """``(values, arg)``: per-segment maximum and its source row."""
    return seg_reduce(src, indptr, "max")


def segment_min_csr(src, indptr):
    """``(values, arg)``: per-segment minimum and its source row."""
    return seg_reduce(src, indptr, "min")


def seg_scan(values, offsets, op: str = "sum", exclusive: bool = False, out=None, stream=None):
    """Segmented scan of ``values`` ([N], uint32 / int32 / float32, CUDA) over
    the segments ``offsets`` ([S+1], int64 or uint32, CUDA) delimits: for a
    row of segment s, the inclusive ``sum`` / ``min`` / ``max`` of the
    segment's rows up to it, or (``exclusive``, sum only) of the rows before
    it; rows in no segment give 0.  Not synchronised."""
    torch = _torch()
    if op not in ("sum", "min", "max"):
        raise ValueError("op must be sum, min or max")
    if exclusive and op != "sum":
        raise ValueError("the exclusive scan is defined for sum")
    if not values.is_cuda or not offsets.is_cuda:
        raise ValueError("values and offsets must be CUDA tensors (there is no CPU path)")
    if values.device != offsets.device:
        raise ValueError("values and offsets must be on the same device")
    if values.dim() != 1 or offsets.dim() != 1 or offsets.numel() < 1:
        raise ValueError("values must be [N] and offsets [S+1]")
    if not values.is_contiguous() or not offsets.is_contiguous():
        raise ValueError("values and offsets must be contiguous")
    n = values.numel()
    if out is None:
        out = torch.empty_like(values)
    elif out.shape != values.shape or out.dtype != values.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like values")
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(values.device)
    with torch.cuda.device(values.device):
        rc = lib.seg_scan(values.data_ptr() if n else None, _value_code(values), n, offsets.data_ptr(),
                          _offset_code(offsets), offsets.numel() - 1, OPS[op], 1 if exclusive else 0,
                          out.data_ptr() if n else None, ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_scan")
    return out


def segment_cumsum_csr(src, indptr):
    """Inclusive per-segment cumulative sum (``seg_scan`` with ``sum``)."""
    return seg_scan(src, indptr, "sum")


def scatter(src, index, dim_size: int, reduce: str = "sum", out=None, out_arg=None,
            with_arg: bool = True, deterministic: bool = False, stream=None):
    """Scatter the rows of ``src`` ([N] or [N, F], CUDA) into ``dim_size``
    outputs named by ``index`` ([N] int64, CUDA) -- graph-reduce README,
    "API": ``sum`` (or ``add``), ``mean`` (float32; 0 where nothing arrived),
    ``max`` / ``min`` returning ``(values, arg)`` (the lowest row holding the
    extreme; 0 and -1 where nothing arrived).  A row whose index is outside
    [0, dim_size) goes nowhere.  float32 sums and means use atomics and are
    not bitwise reproducible unless ``deterministic``: then the rows are
    stably sorted by destination on the device and reduced by the segmented
    path (``seg_scatter_sorted``), so every result repeats bit for bit, at
    the cost of the sort and a gather.  Not synchronised."""
    torch = _torch()
    op = "sum" if reduce == "add" else reduce
    if op not in OPS:
        raise ValueError(f"reduce must be one of {sorted(OPS) + ['add']}")
    if not src.is_cuda or not index.is_cuda:
        raise ValueError("src and index must be CUDA tensors (there is no CPU path)")
    if src.device != index.device:
        raise ValueError("src and index must be on the same device")
    if src.dim() not in (1, 2) or index.dim() != 1 or index.numel() != src.shape[0]:
        raise ValueError("src must be [N] or [N, F] and index [N]")
    if index.dtype != torch.int64:
        raise TypeError("index must be int64")
    if not src.is_contiguous() or not index.is_contiguous():
        raise ValueError("src and index must be contiguous")
    n = src.shape[0]
    feat = 1 if src.dim() == 1 else src.shape[1]
    oshape = (dim_size,) if src.dim() == 1 else (dim_size, feat)
    if out is None:
        out = torch.empty(oshape, dtype=src.dtype, device=src.device)
    elif tuple(out.shape) != oshape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {src.dtype} tensor of shape {oshape}")
    want_arg = op in ("min", "max") and (with_arg or out_arg is not None)
    if want_arg and out_arg is None:
        out_arg = torch.empty(oshape, dtype=torch.int64, device=src.device)
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(src.device)
    fn = lib.seg_scatter_sorted if deterministic else lib.seg_scatter
    with torch.cuda.device(src.device):
        rc = fn(src.data_ptr() if n else None, _value_code(src), feat, n,
                index.data_ptr() if n else None, dim_size, OPS[op],
                out.data_ptr() if dim_size else None,
                out_arg.data_ptr() if (want_arg and dim_size) else None,
                ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_scatter_sorted" if deterministic else "seg_scatter")
    return (out, out_arg) if want_arg else out


def scatter_sum(src, index, dim_size):
    """Sum of the rows sent to each output (graph-reduce README, ``scatter_sum``)."""
    return scatter(src, index, dim_size, "sum")


scatter_add = scatter_sum


def scatter_mean(src, index, dim_size):
    """Mean of the rows sent to each output; 0 where none arrived."""
    return scatter(src, index, dim_size, "mean")


def scatter_max(src, index, dim_size):
    """``(values, argmax)`` over the rows sent to each output."""
    return scatter(src, index, dim_size, "max")


def scatter_min(src, index, dim_size):
    """``(values, argmin)`` over the rows sent to each output."""
    return scatter(src, index, dim_size, "min")


def seg_reduce_sequential(values, offsets, op: str = "sum", out=None, stream=None):
    """The input-order float32 ``sum`` / ``mean`` (graph-reduce README,
    "Correctness": a fixed summation order): out[s, f] starts at 0.0f and
    adds the segment's rows in order, rounding each addition to float32;
    mean divides by the length; empty segments give 0.  ``values`` is
    float32 ``[N]`` or ``[N, F]`` on CUDA.  Slower than ``seg_reduce`` on long
    segments (one dependent addition per row); use it for results that must
    match an in-order float32 loop bit for bit."""
    torch = _torch()
    if op not in ("sum", "mean"):
        raise ValueError("the input-order mode is defined for sum and mean")
    if not values.is_cuda or not offsets.is_cuda:
        raise ValueError("values and offsets must be CUDA tensors (there is no CPU path)")
    if values.dtype != torch.float32:
        raise TypeError("the input-order mode takes float32 values")
    if values.device != offsets.device:
        raise ValueError("values and offsets must be on the same device")
    if values.dim() not in (1, 2) or offsets.dim() != 1 or offsets.numel() < 1:
        raise ValueError("values must be [N] or [N, F] and offsets [S+1]")
    if not values.is_contiguous() or not offsets.is_contiguous():
        raise ValueError("values and offsets must be contiguous")
    n = values.shape[0]
    feat = 1 if values.dim() == 1 else values.shape[1]
    s = offsets.numel() - 1
    oshape = (s,) if values.dim() == 1 else (s, feat)
    if out is None:
        out = torch.empty(oshape, dtype=torch.float32, device=values.device)
    elif tuple(out.shape) != oshape or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous float32 tensor of shape {oshape}")
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(values.device)
    with torch.cuda.device(values.device):
        rc = lib.seg_reduce_sequential(values.data_ptr() if n else None, feat, n, offsets.data_ptr(),
                                       _offset_code(offsets), s, OPS[op], out.data_ptr() if s else None,
                                       ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_reduce_sequential")
    return out


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _out_buffer(t, n, dtype, device, name):
    """A caller's preallocated output (checked) or a new one of n entries."""
    torch = _torch()
    if t is None:
        return torch.empty(n, dtype=dtype, device=device)
    if t.dtype != dtype or t.dim() != 1 or t.numel() < n or not t.is_contiguous() \
            or t.device != device:
        raise ValueError(f"{name} must be a contiguous 1-D {dtype} CUDA tensor of at least {n} entries")
    return t


def seg_rle(keys, values=None, lengths=None, offsets=None, count=None, want_values=True,
            want_lengths=True, want_offsets=True, stream=None):
    """Run-length encode ``keys`` ([n] uint32 or int32, CUDA; equality is on
    the bits) on the device (GPURunLengthEncode / GPUUnique "Contract").

    Returns ``(values, lengths, offsets, count)``: ``values`` (keys' dtype) and
    ``lengths`` (uint32) hold ``n`` entries and ``offsets`` (int64) ``n + 1``,
    of which the first ``count`` (``count + 1`` for offsets) are written;
    ``count`` is a one-element int64 CUDA tensor.  Outputs not wanted are
    ``None`` and are not written.  Nothing is synchronised; ``rle`` and
    ``unique`` read the count and trim.
    """
    torch = _torch()
    u32 = getattr(torch, "uint32", None)
    if not keys.is_cuda:
        raise ValueError("keys must be a CUDA tensor (there is no CPU path)")
    if keys.dim() != 1 or not keys.is_contiguous() or keys.dtype not in (torch.int32, u32):
        raise ValueError("keys must be a contiguous 1-D uint32 or int32 tensor")
    n = keys.numel()
    dev = keys.device
    values = _out_buffer(values, n, keys.dtype, dev, "values") if want_values else None
    lengths = _out_buffer(lengths, n, u32, dev, "lengths") if want_lengths else None
    offsets = _out_buffer(offsets, n + 1, torch.int64, dev, "offsets") if want_offsets else None
    count = _out_buffer(count, 1, torch.int64, dev, "count")
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.seg_rle(keys.data_ptr() if n else None, n, _ptr(values), _ptr(lengths),
                         _ptr(offsets), count.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_rle")
    return values, lengths, offsets, count


def rle(keys):
    """``(values, lengths, offsets)`` of the runs of ``keys``, trimmed to the
    run count (reads the count back, so it synchronises)."""
    values, lengths, offsets, count = seg_rle(keys)
    c = int(count.item())
    return values[:c], lengths[:c], offsets[:c + 1]


def unique(keys):
    """The first key of every run of equal adjacent keys (GPUUnique), trimmed
    to the run count (synchronises)."""
    values, _, _, count = seg_rle(keys, want_lengths=False, want_offsets=False)
    return values[:int(count.item())]


def seg_flags_to_offsets(flags, offsets=None, count=None, stream=None):
    """Offsets from segment-start ``flags`` ([n] uint8 or bool, CUDA):
    every index with a non-zero flag starts a segment; the offsets list those
    indices, then n (GPUSegmentedLayout).  Returns ``(offsets, count)`` with
    ``offsets`` of ``n + 1`` int64 entries, the first ``count + 1`` written;
    not synchronised."""
    torch = _torch()
    if not flags.is_cuda:
        raise ValueError("flags must be a CUDA tensor (there is no CPU path)")
    if flags.dim() != 1 or not flags.is_contiguous() or flags.dtype not in (torch.uint8, torch.bool):
        raise ValueError("flags must be a contiguous 1-D uint8 or bool tensor")
    n = flags.numel()
    dev = flags.device
    offsets = _out_buffer(offsets, n + 1, torch.int64, dev, "offsets")
    count = _out_buffer(count, 1, torch.int64, dev, "count")
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.seg_flags_to_offsets(flags.data_ptr() if n else None, n, offsets.data_ptr(),
                                      count.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_flags_to_offsets")
    return offsets, count


def flags_to_offsets(flags):
    """``seg_flags_to_offsets`` trimmed to ``count + 1`` entries (synchronises)."""
    offsets, count = seg_flags_to_offsets(flags)
    return offsets[:int(count.item()) + 1]


def selftest_wait_timeout(limit_ms: int = 50, stream=None) -> None:
    """Launch the library's self-test of its bounded waits: a wait on a
    phase that nothing completes, which runs out after ``limit_ms`` and
    records a timeout in the device status word (read it with
    ``device_status()``)."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = load_library().seg_selftest_wait_timeout(limit_ms, ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise SegReduceError(rc, "seg_selftest_wait_timeout")


def device_status(stream=None) -> int:
    """Synchronise ``stream`` and read (and clear) the device status word:
    0 if no kernel on the current device recorded a timed-out wait."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return load_library().seg_reduce_device_status(ctypes.c_void_p(stream.cuda_stream))
