"""Seeded synthetic inputs for segmented reduction over CSR offsets.

This module only draws inputs and counts bytes; it holds none of the
reduction's arithmetic, and both the CUDA path (through its tests and the
benchmark) and the CPU oracle consume what it returns.

Five workloads, each a fixed recipe drawn from ``numpy.random.Generator(PCG64)``
with seed ``20261202 + index``:

=========  ===================================================================
tiny       1,000 segments, lengths uniform in [0, 16] with 5% forced empty,
           uint32 offsets; float32 U[-1, 1) and uint32 U[0, 2^16) values.
bulk       1,000,000 segments, lengths geometric (mean 16, >= 1), int64
           offsets; int32 U[-2^20, 2^20], uint32 = the same bits, float32
           N(0, 1).
mp         message passing: 1,000,000 rows x 64 float32 N(0, 1); each row's
           destination uniform over 10,000 segments, rows in destination
           order, indptr = [0] + cumsum(bincount) (graph-reduce README,
           "Usage"), int64.
skewed     64,000,000 float32 N(0, 1) over 1,000,000 segments: 200,000 empty
           at random positions, 4 giants of 6.0M / 5.5M / 5.2M / 5.1M rows at
           random positions, the rest Zipf(1.5) clipped at 1M and scaled to
           42.2M rows in total (largest remainder, each >= 1); int64.
large      10,000,000 rows x 128 float32 N(0, 1) over 100,000 segments with
           power-law lengths (floor(Pareto(1.1) + 1), clipped at 10M, scaled
           to 10M rows, each >= 1); int64.
=========  ===================================================================

``large_1m`` is the large recipe at a tenth of the size (1,000,000 rows x
128 over 10,000 segments, seed ``20261202 + 50``): a case small enough for
hardware-counter captures of the large workload's kernel shape.

The mp workload draws i.i.d. rows directly in destination order: permuting
i.i.d. rows by a stable sort of their destinations gives the same
distribution, so the sort is not materialised.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
NAMES = ("tiny", "bulk", "mp", "skewed", "large")

_BLOCK = 1 << 22          # values are filled in fixed blocks, each with its own stream


@dataclass
class Workload:
    name: str
    offsets: np.ndarray                       # [S+1], uint32 or int64
    values: dict = field(default_factory=dict)  # dtype name -> [N] or [N, F]
    feat: int = 1
    cases: tuple = ()                         # (dtype name, op) pairs run on it
    seed: int = 0

    @property
    def num_segments(self) -> int:
        return int(self.offsets.shape[0] - 1)

    @property
    def num_rows(self) -> int:
        return int(next(iter(self.values.values())).shape[0])


def algorithmic_bytes(num_rows: int, feat: int, num_segments: int,
                      offset_itemsize: int, op: str) -> int:
    """Minimum bytes one reduction moves: values read + offsets read +
    outputs written + int64 args written (min / max only)."""
    b = num_rows * feat * 4 + (num_segments + 1) * offset_itemsize
    b += num_segments * feat * 4
    if op in ("min", "max"):
        b += num_segments * feat * 8
    return b


def workload_bytes(w: Workload, dtype: str, op: str) -> int:
    return algorithmic_bytes(w.num_rows, w.feat, w.num_segments,
                             w.offsets.dtype.itemsize, op)


def offsets_from_lengths(lengths, dtype=np.int64) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    return off.astype(dtype)


def scale_to_total(weights, total: int) -> np.ndarray:
    """Integers >= 1 summing to ``total`` in proportion to ``weights``
    (largest-remainder rounding, ties broken by index)."""
    w = np.asarray(weights, dtype=np.float64)
    n = w.shape[0]
    spare = total - n
    if spare < 0:
        raise ValueError("total smaller than the number of parts")
    q = spare * w / w.sum()
    base = np.floor(q).astype(np.int64)
    rest = spare - int(base.sum())
    frac = q - base
    order = np.lexsort((np.arange(n), -frac))   # largest fraction first, then index
    base[order[:rest]] += 1
    return base + 1


def _fill_values(shape, seed: int, kind: str, lo=None, hi=None) -> np.ndarray:
    """Fill an array block by block; block k uses SeedSequence(seed).spawn()[k],
    so the result does not depend on how many threads fill it."""
    out_dtype = {"normal": np.float32, "uniform": np.float32,
                 "u32": np.uint32, "s32": np.int32}[kind]
    a = np.empty(int(np.prod(shape)), dtype=out_dtype)
    nblocks = (a.shape[0] + _BLOCK - 1) // _BLOCK
    seqs = np.random.SeedSequence(seed).spawn(max(nblocks, 1))

    def work(k):
        rng = np.random.Generator(np.random.PCG64(seqs[k]))
        sl = a[k * _BLOCK:(k + 1) * _BLOCK]
        if kind == "normal":
            rng.standard_normal(out=sl, dtype=np.float32)
        elif kind == "uniform":
            sl[:] = rng.uniform(lo, hi, size=sl.shape[0]).astype(np.float32)
        elif kind == "u32":
            sl[:] = rng.integers(lo, hi, size=sl.shape[0], dtype=np.uint32)
        else:
            sl[:] = rng.integers(lo, hi, size=sl.shape[0], dtype=np.int32,
                                 endpoint=True)

    workers = max(1, min(16, os.cpu_count() or 1))
    if nblocks <= 1:
        work(0)
    else:
        with _cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(work, range(nblocks)))
    return a.reshape(shape)


def make(name: str, with_values: bool = True) -> Workload:
    """Draw workload ``name``; ``with_values=False`` draws only the offsets
    (the values then hold zero-row placeholders of the right dtype)."""
    idx = NAMES.index(name) if name in NAMES else None
    seed = SEED_BASE + (idx if idx is not None else 50)
    rng = np.random.Generator(np.random.PCG64(seed))

    def _fill(shape, sd, kind, lo=None, hi=None):
        if not with_values:
            return np.empty((0,) + tuple(shape[1:]), dtype={"normal": np.float32,
                            "uniform": np.float32, "u32": np.uint32, "s32": np.int32}[kind])
        return _fill_values(shape, sd, kind, lo, hi)
    if name == "tiny":
        S = 1000
        lengths = rng.integers(0, 16, size=S, endpoint=True)
        lengths[rng.choice(S, size=S // 20, replace=False)] = 0
        off = offsets_from_lengths(lengths, np.uint32)
        n = int(off[-1])
        vals = {"f32": _fill((n,), seed + 1000, "uniform", -1.0, 1.0),
                "u32": _fill((n,), seed + 2000, "u32", 0, 1 << 16)}
        cases = tuple((d, op) for d in ("f32", "u32") for op in ("sum", "min", "max"))
        return Workload(name, off, vals, 1, cases, seed)
    if name == "bulk":
        S = 1_000_000
        lengths = rng.geometric(1.0 / 16.0, size=S)
        off = offsets_from_lengths(lengths)
        n = int(off[-1])
        s32 = _fill((n,), seed + 1000, "s32", -(1 << 20), 1 << 20)
        vals = {"u32": s32.view(np.uint32), "s32": s32,
                "f32": _fill((n,), seed + 2000, "normal")}
        cases = tuple((d, op) for d in ("u32", "s32", "f32")
                      for op in ("sum", "min", "max"))
        return Workload(name, off, vals, 1, cases, seed)
    if name == "mp":
        N, F, S = 1_000_000, 64, 10_000
        dst = rng.integers(0, S, size=N)
        off = offsets_from_lengths(np.bincount(dst, minlength=S))
        vals = {"f32": _fill((N, F), seed + 1000, "normal")}
        return Workload(name, off, vals, F, (("f32", "sum"), ("f32", "mean"),
                                             ("f32", "max")), seed)
    if name == "skewed":
        N, S = 64_000_000, 1_000_000
        giants = np.array([6_000_000, 5_500_000, 5_200_000, 5_100_000], np.int64)
        pos = rng.permutation(S)
        empty_pos = pos[:200_000]
        giant_pos = pos[200_000:200_004]
        rest_pos = np.sort(pos[200_004:])
        draws = np.minimum(rng.zipf(1.5, size=rest_pos.shape[0]), 1_000_000)
        lengths = np.zeros(S, dtype=np.int64)
        lengths[giant_pos] = giants
        lengths[rest_pos] = scale_to_total(draws, N - int(giants.sum()))
        lengths[empty_pos] = 0
        off = offsets_from_lengths(lengths)
        vals = {"f32": _fill((N,), seed + 1000, "normal")}
        return Workload(name, off, vals, 1, tuple(("f32", op) for op in
                                                  ("sum", "min", "max")), seed)
    if name in ("large", "large_1m"):
        N, F, S = (10_000_000, 128, 100_000) if name == "large" else (1_000_000, 128, 10_000)
        draws = np.minimum(np.floor(rng.pareto(1.1, size=S) + 1.0), N)
        off = offsets_from_lengths(scale_to_total(draws, N))
        vals = {"f32": _fill((N, F), seed + 1000, "normal")}
        return Workload(name, off, vals, F, (("f32", "sum"), ("f32", "max")), seed)
    raise KeyError(name)


def random_offsets(rng, num_rows: int, num_segments: int, empty_frac=0.1,
                   dtype=np.int64, start=0, stop=None) -> np.ndarray:
    """Random nondecreasing offsets over rows [start, stop) (test helper)."""
    stop = num_rows if stop is None else stop
    if num_segments == 0:
        return np.array([start], dtype=dtype)
    cuts = np.sort(rng.integers(start, stop + 1, size=num_segments - 1))
    off = np.concatenate([[start], cuts, [stop]]).astype(np.int64)
    if empty_frac > 0 and num_segments > 2:
        k = int(empty_frac * num_segments)
        idx = rng.choice(np.arange(1, num_segments), size=k, replace=False)
        off[idx] = off[idx - 1]
        off = np.maximum.accumulate(off)
    return off.astype(dtype)


def stats(w: Workload) -> dict:
    lengths = np.diff(w.offsets.astype(np.int64))
    return {"name": w.name, "rows": w.num_rows, "feat": w.feat,
            "segments": w.num_segments, "empty": int((lengths == 0).sum()),
            "max_len": int(lengths.max()) if lengths.size else 0,
            "over_5M": int((lengths > 5_000_000).sum())}


# ---- inputs of the offsets producers (run-length encoding, flags) ----------

def segment_keys(offsets: np.ndarray) -> np.ndarray:
    """The ordered uint32 key of every row: the id of the segment it falls in
    (rows before offsets[0] get key 0).  This is the sorted-keys input that
    run-length encoding turns back into the offsets of the non-empty
    segments ("sorted keys -> run-length encode -> segment metadata")."""
    off = offsets.astype(np.int64)
    keys = np.zeros(int(off[-1]), dtype=np.uint32)
    lengths = np.diff(off)
    keys[int(off[0]):] = np.repeat(np.arange(lengths.shape[0], dtype=np.uint32), lengths)
    return keys


def segment_flags(offsets: np.ndarray) -> np.ndarray:
    """uint8 flags over rows [0, offsets[-1]): 1 where a non-empty segment starts."""
    off = offsets.astype(np.int64)
    flags = np.zeros(int(off[-1]), dtype=np.uint8)
    starts = off[:-1][np.diff(off) > 0]
    flags[starts] = 1
    return flags


def random_runs(n: int, mean_run: float, seed: int, distinct: int = 1 << 32) -> np.ndarray:
    """n uint32 keys made of runs with geometric lengths (mean ``mean_run``),
    each run's key drawn uniformly from [0, distinct).  Neighbouring runs may
    draw the same key, which merges them (as it should)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if n == 0:
        return np.zeros(0, dtype=np.uint32)
    lens = rng.geometric(1.0 / mean_run, size=int(n / mean_run) + 16)
    while lens.sum() < n:
        lens = np.concatenate([lens, rng.geometric(1.0 / mean_run, size=lens.shape[0])])
    keys = rng.integers(0, distinct, size=lens.shape[0], dtype=np.uint64).astype(np.uint32)
    return np.repeat(keys, lens)[:n]


def random_flags(n: int, p: float, seed: int) -> np.ndarray:
    """n uint8 flags, each non-zero with probability p (non-zero values vary)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    on = rng.random(n) < p
    return np.where(on, rng.integers(1, 256, size=n), 0).astype(np.uint8)



# ---- input of the unsorted scatter path -----------------------------------

def scatter_input(name: str = "mp"):
    """(src, index, dim_size) for the scatter path: the message-passing shape
    of the graph-reduce README "Measured" table -- 1,000,000 float32 rows of
    64 (``mp``) or 16 (``mp16``) columns, N(0, 1), each sent to an output
    drawn uniformly from 10,000, in no particular order."""
    feat = {"mp": 64, "mp16": 16}[name]
    seed = SEED_BASE + 100 + feat
    rng = np.random.Generator(np.random.PCG64(seed))
    index = rng.integers(0, 10_000, size=1_000_000).astype(np.int64)
    src = _fill_values((1_000_000, feat), seed + 1, "normal")
    return src, index, 10_000
