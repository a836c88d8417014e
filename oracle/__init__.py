"""CPU oracle for segmented reduction over offset-delimited (CSR) segments.

TEST INFRASTRUCTURE ONLY.  The product path never imports this package: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may.  It shares no code with the CUDA library.

Two independent implementations live here:

* ``seg_reduce``: the sequential C loop in ``seg_oracle.c`` (built with gcc,
  called through ctypes) -- the oracle proper, fast enough for the full
  synthetic workloads.
* ``seg_reduce_parallel``: the same C loop built a second time with OpenMP
  over (segment, column) pairs, for the benchmark's all-cores CPU baseline
  only (each output is computed exactly as in the sequential build).
* ``brute.seg_reduce``: a pure-Python restatement with Python integers and
  ``math.fsum`` for tiny inputs, used to pin the C oracle.
* ``seg_reduce_sequential``: the input-order float32 sum / mean of
  ``seq_oracle.c`` (graph-reduce README, "Correctness": the fixed summation
  order of ``torch.segment_reduce``), pinned by ``brute.seg_reduce_sequential``.
* ``scatter``: the unsorted scatter of ``scatter_oracle.c`` (graph-reduce
  README, "API"), pinned against ``seg_reduce`` after a stable sort of the
  index and against ``brute.scatter``.
* ``seg_scan``: the segmented inclusive / exclusive scan of
  ``scan_oracle.c``, pinned against ``seg_reduce`` (every prefix is a
  reduction), numpy's cumulative routines per segment and ``brute.seg_scan``.
* ``rle`` / ``flags_to_offsets``: the sequential C loops in ``rle_oracle.c``
  for the producers of offsets (GPURunLengthEncode / GPUUnique,
  GPUSegmentedLayout), pinned by ``brute.rle`` / ``brute.flags_to_offsets``.

Semantics (GPUSegmentedReduction "Contract"; graph-reduce README "API",
"Method" and "Correctness"): segment ``s`` reduces rows
``[offsets[s], offsets[s+1])`` of ``values`` (shape ``[N]`` or ``[N, F]``,
reduced over dimension 0); ops ``sum``, ``min``, ``max`` for uint32 / int32 /
float32 and ``mean`` for float32; ``min``/``max`` also give the absolute source
row (ties to the lower row); empty segments give 0 and arg -1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "seg_oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "libsegoracle.so")
_RLE_SRC = os.path.join(_HERE, "rle_oracle.c")
_RLE_LIB = os.path.join(_LIBDIR, "libsegrleoracle.so")
_SCATTER_SRC = os.path.join(_HERE, "scatter_oracle.c")
_SCATTER_LIB = os.path.join(_LIBDIR, "libsegscatteroracle.so")
_SCAN_SRC = os.path.join(_HERE, "scan_oracle.c")
_SCAN_LIB = os.path.join(_LIBDIR, "libsegscanoracle.so")
_SEQ_SRC = os.path.join(_HERE, "seq_oracle.c")
_SEQ_LIB = os.path.join(_LIBDIR, "libsegseqoracle.so")
_PAR_LIB = os.path.join(_LIBDIR, "libsegoracle_par.so")

# Codes private to seg_oracle.c.
_DT = {np.dtype(np.uint32): 0, np.dtype(np.int32): 1, np.dtype(np.float32): 2}
_OFF = {np.dtype(np.uint32): 0, np.dtype(np.int64): 1}
_OP = {"sum": 0, "min": 1, "max": 2, "mean": 3}
_ERR = {-1: "bad argument", -2: "offsets not nondecreasing within [0, N]",
        -3: "mean is defined for float32 only"}

_lock = threading.Lock()
_lib = None


def compile_source(src: str, dst: str, extra=()) -> str:
    """gcc -O2 without fast-math or FMA contraction, as a shared library."""
    tmp = dst + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", *extra, "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, dst)
    return dst


def build(force: bool = False) -> str:
    """Compile seg_oracle.c into lib/libsegoracle.so, rle_oracle.c into
    lib/libsegrleoracle.so, seq_oracle.c into lib/libsegseqoracle.so and
    scatter_oracle.c into lib/libsegscatteroracle.so and scan_oracle.c into
    lib/libsegscanoracle.so."""
    os.makedirs(_LIBDIR, exist_ok=True)
    for src, lib in ((_RLE_SRC, _RLE_LIB), (_SEQ_SRC, _SEQ_LIB), (_SCATTER_SRC, _SCATTER_LIB),
                     (_SCAN_SRC, _SCAN_LIB), (_SRC, _LIB)):
        if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
            compile_source(src, lib)
    return _LIB


def load_library(path: str):
    """ctypes handle of a compiled oracle library (the default one, or a
    deliberately broken copy that a test builds to check the pins)."""
    lib = ctypes.CDLL(path)
    lib.oracle_seg_reduce.restype = ctypes.c_int
    lib.oracle_seg_reduce.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    return lib


_par_lib = None


def load_parallel_library():
    """The all-cores build of seg_oracle.c (OpenMP over (segment, column)
    pairs), compiled on first use; raises if gcc has no OpenMP."""
    global _par_lib
    with _lock:
        if _par_lib is None:
            os.makedirs(_LIBDIR, exist_ok=True)
            if not os.path.exists(_PAR_LIB) or os.path.getmtime(_PAR_LIB) < os.path.getmtime(_SRC):
                compile_source(_SRC, _PAR_LIB, ("-fopenmp", "-DORC_PARALLEL_SEGMENTS"))
            _par_lib = load_library(_PAR_LIB)
    return _par_lib


def parallel_threads() -> int:
    """Threads the all-cores build runs on (OMP_NUM_THREADS, else every core)."""
    return int(load_parallel_library().oracle_threads())


def seg_reduce_parallel(values, offsets, op: str, with_arg: bool = True):
    """``seg_reduce`` through the all-cores build: the same outputs, bit for bit."""
    return seg_reduce(values, offsets, op, with_arg=with_arg, lib=load_parallel_library())


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB)
    return _lib


def seg_reduce(values, offsets, op: str, with_arg: bool = True, lib=None):
    """Reduce ``values`` ([N] or [N, F]) over the segments that ``offsets`` ([S+1]) delimits.

    Returns ``out`` (shape ``[S]`` or ``[S, F]``, dtype of ``values``) for
    sum / mean, and ``(out, arg)`` (arg int64, same shape) for min / max
    when ``with_arg``.
    """
    values = np.ascontiguousarray(values)
    offsets = np.ascontiguousarray(offsets)
    if values.dtype not in _DT:
        raise TypeError(f"unsupported values dtype {values.dtype}")
    if offsets.dtype not in _OFF:
        raise TypeError(f"unsupported offsets dtype {offsets.dtype}")
    if op not in _OP:
        raise ValueError(f"unknown op {op!r}")
    if values.ndim not in (1, 2) or offsets.ndim != 1 or offsets.shape[0] < 1:
        raise ValueError("values must be [N] or [N, F]; offsets must be [S+1]")
    n = values.shape[0]
    f = 1 if values.ndim == 1 else values.shape[1]
    s = offsets.shape[0] - 1
    oshape = (s,) if values.ndim == 1 else (s, f)
    out = np.zeros(oshape, dtype=values.dtype)
    want_arg = with_arg and op in ("min", "max")
    arg = np.zeros(oshape, dtype=np.int64) if want_arg else None
    lib = _load() if lib is None else lib
    rc = lib.oracle_seg_reduce(
        values.ctypes.data, _DT[values.dtype], f, n,
        offsets.ctypes.data, _OFF[offsets.dtype], s, _OP[op],
        out.ctypes.data, arg.ctypes.data if want_arg else None)
    if rc != 0:
        raise ValueError(f"oracle rejected the input: {_ERR.get(rc, rc)}")
    return (out, arg) if want_arg else out



_rle_lib = None


def load_rle_library(path: str):
    """ctypes handle of a compiled RLE oracle library (the default one, or a
    deliberately broken copy that a test builds to check the pins)."""
    lib = ctypes.CDLL(path)
    lib.oracle_rle.restype = ctypes.c_int64
    lib.oracle_rle.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p]
    lib.oracle_flags_to_offsets.restype = ctypes.c_int64
    lib.oracle_flags_to_offsets.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    return lib


def _load_rle():
    global _rle_lib
    with _lock:
        if _rle_lib is None:
            build()
            _rle_lib = load_rle_library(_RLE_LIB)
    return _rle_lib


def rle(keys, lib=None):
    """Run-length encoding of an ordered uint32 vector: ``(values, lengths,
    offsets)`` with ``offsets`` one longer (run starts, then n)."""
    keys = np.ascontiguousarray(keys, dtype=np.uint32)
    n = keys.shape[0]
    values = np.zeros(n, np.uint32)
    lengths = np.zeros(n, np.uint32)
    offsets = np.zeros(n + 1, np.int64)
    lib = _load_rle() if lib is None else lib
    runs = lib.oracle_rle(keys.ctypes.data if n else None, n, values.ctypes.data, lengths.ctypes.data,
                          offsets.ctypes.data)
    if runs < 0:
        raise ValueError("oracle rejected the input")
    return values[:runs].copy(), lengths[:runs].copy(), offsets[: runs + 1].copy()


def flags_to_offsets(flags, lib=None):
    """Offsets from segment-start flags: the indices of the non-zero flags, then n."""
    flags = np.ascontiguousarray(flags, dtype=np.uint8)
    n = flags.shape[0]
    offsets = np.zeros(n + 1, np.int64)
    lib = _load_rle() if lib is None else lib
    count = lib.oracle_flags_to_offsets(flags.ctypes.data if n else None, n, offsets.ctypes.data)
    if count < 0:
        raise ValueError("oracle rejected the input")
    return offsets[: count + 1].copy()


_seq_lib = None


def load_seq_library(path: str):
    """ctypes handle of a compiled sequential-sum oracle (the default one, or
    a deliberately broken copy that a test builds to check the pins)."""
    lib = ctypes.CDLL(path)
    lib.oracle_seg_sequential_f32.restype = ctypes.c_int
    lib.oracle_seg_sequential_f32.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                              ctypes.c_void_p]
    return lib


def _load_seq():
    global _seq_lib
    with _lock:
        if _seq_lib is None:
            build()
            _seq_lib = load_seq_library(_SEQ_LIB)
    return _seq_lib


def seg_reduce_sequential(values, offsets, op: str = "sum", lib=None):
    """Input-order float32 ``sum`` or ``mean`` of ``values`` ([N] or [N, F]
    float32) over the segments ``offsets`` ([S+1]) delimits: each sum starts
    at 0.0f and adds the rows in order, rounding every addition to float32."""
    if op not in ("sum", "mean"):
        raise ValueError("the input-order mode is defined for sum and mean")
    values = np.ascontiguousarray(values, dtype=np.float32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    n = values.shape[0]
    feat = 1 if values.ndim == 1 else int(np.prod(values.shape[1:]))
    s = offsets.shape[0] - 1
    out = np.zeros((s,) + values.shape[1:], dtype=np.float32)
    lib = _load_seq() if lib is None else lib
    rc = lib.oracle_seg_sequential_f32(values.ctypes.data if n else None, n, feat,
                                       offsets.ctypes.data, s, 1 if op == "mean" else 0,
                                       out.ctypes.data if s else None)
    if rc != 0:
        raise ValueError({-1: "bad argument", -2: "offsets not nondecreasing within [0, N]"}.get(rc, rc))
    return out


_scatter_lib = None


def load_scatter_library(path: str):
    """ctypes handle of a compiled scatter oracle (the default one, or a
    deliberately broken copy that a test builds to check the pins)."""
    lib = ctypes.CDLL(path)
    lib.oracle_scatter.restype = ctypes.c_int
    lib.oracle_scatter.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                   ctypes.c_void_p]
    return lib


def _load_scatter():
    global _scatter_lib
    with _lock:
        if _scatter_lib is None:
            build()
            _scatter_lib = load_scatter_library(_SCATTER_LIB)
    return _scatter_lib


def scatter(src, index, dim_size: int, op: str, with_arg: bool = True, lib=None):
    """Scatter the rows of ``src`` ([N] or [N, F]) into ``dim_size`` outputs
    named by ``index`` ([N] int64): ``sum`` / ``mean`` / ``min`` / ``max``.
    Returns ``out`` or ``(out, arg)`` for min / max."""
    src = np.ascontiguousarray(src)
    if src.dtype not in _DT:
        raise TypeError(f"unsupported dtype {src.dtype}")
    index = np.ascontiguousarray(index, dtype=np.int64)
    n = src.shape[0]
    feat = 1 if src.ndim == 1 else int(np.prod(src.shape[1:]))
    if index.shape != (n,):
        raise ValueError("index must be [N]")
    shape = (dim_size,) + src.shape[1:]
    out = np.zeros(shape, dtype=src.dtype)
    arg = np.full(shape, -1, dtype=np.int64) if op in ("min", "max") else None
    lib = _load_scatter() if lib is None else lib
    rc = lib.oracle_scatter(src.ctypes.data if n else None, _DT[src.dtype], feat, n,
                            index.ctypes.data if n else None, dim_size, _OP[op],
                            out.ctypes.data if dim_size else None,
                            arg.ctypes.data if (arg is not None and dim_size) else None)
    if rc != 0:
        raise ValueError({-1: "bad argument", -3: "mean is defined for float32 only",
                          -4: "out of memory"}.get(rc, rc))
    if arg is not None and with_arg:
        return out, arg
    return out


_scan_lib = None


def load_scan_library(path: str):
    """ctypes handle of a compiled scan oracle (the default one, or a
    deliberately broken copy that a test builds to check the pins)."""
    lib = ctypes.CDLL(path)
    lib.oracle_seg_scan.restype = ctypes.c_int
    lib.oracle_seg_scan.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return lib


def _load_scan():
    global _scan_lib
    with _lock:
        if _scan_lib is None:
            build()
            _scan_lib = load_scan_library(_SCAN_LIB)
    return _scan_lib


def seg_scan(values, offsets, op: str = "sum", exclusive: bool = False, lib=None):
    """Segmented scan of ``values`` ([N], uint32 / int32 / float32) over the
    segments ``offsets`` ([S+1]) delimits; rows in no segment give 0."""
    values = np.ascontiguousarray(values)
    if values.dtype not in _DT or values.ndim != 1:
        raise TypeError("values must be a 1-D uint32, int32 or float32 array")
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    n = values.shape[0]
    out = np.empty(n, dtype=values.dtype)
    lib = _load_scan() if lib is None else lib
    rc = lib.oracle_seg_scan(values.ctypes.data if n else None, _DT[values.dtype], n,
                             offsets.ctypes.data, offsets.shape[0] - 1, _OP[op], 1 if exclusive else 0,
                             out.ctypes.data if n else None)
    if rc != 0:
        raise ValueError({-1: "bad argument", -2: "offsets not nondecreasing within [0, N]"}.get(rc, rc))
    return out
