"""Pure-Python brute force of segmented reduction, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It is written
independently of ``seg_oracle.c`` so that each pins the other: Python integers
reduced modulo 2**32 for integer sums, ``math.fsum`` (the correctly rounded
sum) for float sums, and an explicit loop that keeps the first row holding
the extreme for min / max (graph-reduce README, "Method": ties go to the
lower row).  Segment semantics follow GPUSegmentedReduction, "What is an
offset-delimited segment?" and "Contract".
"""
from __future__ import annotations

import math
import struct

import numpy as np


def _to_f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def _wrap(x: int, signed: bool) -> int:
    x %= 1 << 32
    if signed and x >= 1 << 31:
        x -= 1 << 32
    return x


def seg_reduce(values, offsets, op: str, kind: str, feat=None):
    """``values``: list of rows (each row a list of F numbers), ``offsets``: list of ints.

    ``kind`` is "u32", "s32" or "f32"; ``feat`` (F) is needed when there
    are no rows.  Returns (out, arg): lists of rows;
    arg rows hold -1 for empty segments and for sum / mean.
    """
    S = len(offsets) - 1
    F = feat if feat is not None else (len(values[0]) if values else 1)
    out, arg = [], []
    for s in range(S):
        b, e = offsets[s], offsets[s + 1]
        orow, arow = [], []
        for f in range(F):
            col = [values[r][f] for r in range(b, e)]
            if not col:
                orow.append(0.0 if kind == "f32" else 0)
                arow.append(-1)
                continue
            if op in ("sum", "mean"):
                if kind == "f32":
                    total = _to_f32(math.fsum(col))
                    if op == "mean":
                        total = _to_f32(total / _to_f32(float(len(col))))
                    orow.append(total)
                else:
                    orow.append(_wrap(sum(int(x) for x in col), kind == "s32"))
                arow.append(-1)
            else:
                best_i = 0
                for i in range(1, len(col)):
                    better = col[i] < col[best_i] if op == "min" else col[i] > col[best_i]
                    if better:
                        best_i = i
                orow.append(col[best_i])
                arow.append(b + best_i)
        out.append(orow)
        arg.append(arow)
    return out, arg


def rle(keys):
    """Runs of adjacent equal values by itertools.groupby (GPURunLengthEncode,
    "What is run-length encoding?"): (values, lengths, offsets)."""
    import itertools
    values, lengths, offsets = [], [], []
    pos = 0
    for key, grp in itertools.groupby(list(keys)):
        k = len(list(grp))
        values.append(key)
        lengths.append(k)
        offsets.append(pos)
        pos += k
    offsets.append(pos)
    return values, lengths, offsets


def flags_to_offsets(flags):
    """The indices whose flag is set, then the length (GPUSegmentedLayout)."""
    flags = list(flags)
    return [i for i, f in enumerate(flags) if f] + [len(flags)]


def seg_reduce_sequential(values, offsets, op="sum"):
    """Input-order float32 fold from 0 with numpy float32 scalars, one
    rounded addition per row (graph-reduce README, "Correctness": fixed
    summation order); mean divides the float32 sum by the length."""
    v = np.asarray(values, dtype=np.float32)
    v2 = v.reshape(v.shape[0], -1)
    off = [int(x) for x in offsets]
    out = np.zeros((len(off) - 1, v2.shape[1]), dtype=np.float32)
    for s in range(len(off) - 1):
        b, e = off[s], off[s + 1]
        for f in range(v2.shape[1]):
            acc = np.float32(0.0)
            for r in range(b, e):
                acc = np.float32(acc + v2[r, f])
            if op == "mean":
                acc = np.float32(acc / np.float32(e - b)) if e > b else np.float32(0.0)
            out[s, f] = acc
    return out.reshape((len(off) - 1,) + v.shape[1:])


def scatter(src, index, dim_size, op, kind, feat):
    """Row-by-row scatter (graph-reduce README, "API"): gather each
    destination's rows in row order, then reduce them as one segment with
    ``seg_reduce`` above.  ``src``: list of rows (each a list of F numbers).
    Returns (out, arg) as lists of rows; an index outside [0, dim_size) is
    skipped."""
    groups = [[] for _ in range(dim_size)]
    for r, d in enumerate(index):
        if 0 <= int(d) < dim_size:
            groups[int(d)].append(r)
    outs, args = [], []
    for rows in groups:
        o, a = seg_reduce([src[r] for r in rows], [0, len(rows)], op, kind, feat)
        outs.append(o[0])
        args.append([rows[k] if k >= 0 else -1 for k in a[0]])
    return outs, args


def seg_scan(values, offsets, op, kind, exclusive=False):
    """Every prefix of every segment reduced by ``seg_reduce`` above (one
    segment per prefix): out[r] for offsets[s] <= r < offsets[s+1] is the
    reduction of values[offsets[s] .. r] (.. r - 1 when exclusive, sum only);
    rows in no segment are 0."""
    values = list(values)
    out = [0.0 if kind == "f32" else 0] * len(values)
    off = [int(x) for x in offsets]
    for s in range(len(off) - 1):
        for r in range(off[s], off[s + 1]):
            end = r if exclusive else r + 1
            rows = [[values[i]] for i in range(off[s], end)]
            o, _ = seg_reduce(rows, [0, len(rows)], op, kind, 1)
            out[r] = o[0][0]
    return out
