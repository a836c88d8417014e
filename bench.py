"""Benchmark: segmented reduction over CSR offsets on one GB300 (or N replicas).

A step is one pass of the whole path over the workload: every (dtype, op)
case the workload lists (the scalar-bulk workload: uint32 / int32 / float32
x sum / min+arg / max+arg), each one seg_reduce call = one kernel launch.

value        algorithmic bytes of the step / summed CUDA-event kernel time,
             inputs resident in HBM, L2 flushed before every call, outside
             the events: a 2 x L2 write (no input line stays in L2), then a
             2 x L2 read, so that the call starts from clean lines and does
             not pay for writing back the flush's dirty ones.
e2e          the same bytes / time of a step that copies its inputs from
             pinned host memory, runs the calls and copies the outputs back.
roofline     the reduction kernel against the measured HBM copy bandwidth.
cpu_baseline the C oracle on the host cores (one thread) over the same cases.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

With --producer rle|unique|flags the step is instead one call of that
offsets producer over the ordered segment keys (rle, unique) or segment-start
flags (flags) of the bulk or skewed workload: the input that the producer
turns back into the workload's offsets.  Its line carries the same keys.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "segmented-reduce effective HBM GB/s and % of GB300 peak; segments/s (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
# what shapes the reduction's launches: its kernels and its host planner
KERNEL_SOURCES = ["ptx.cuh", "seg_common.cuh", "seg_rows2.cuh", "seg_scalar.cuh", "seg_small.cuh", "seg_pick.cuh",
                  "seg_plan.cuh", "seg_f32.cu", "seg_u32.cu", "seg_s32.cu"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "segmented_reduction_csr_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(config: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; otherwise None."""
    p = os.path.join(ROOT, "profiles", f"seg_reduce_{config}_traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except Exception:
        return None
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


class L2Flush:
    """Evict the inputs from L2 before a timed call: write a buffer of
    2 x L2, then read two others of 2 x L2 each, so that L2 holds clean lines
    that belong to no input (the clean-cache state that ncu's cache control
    also gives a profiled launch).  One read pass after the write is not
    enough on GB300: the write's last dirty lines are still being written
    back when the timed call starts, and that traffic lands in its time
    (message-passing sum: 56.3 us after one read pass, 51.4 us after two,
    51.5 us when nothing is written at all)."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.r2 = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)
        torch.sum(self.r2, dim=0, out=self.sink)


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- ranks: one process per GPU under torchrun, each an independent replica ---------
def dist_init(backend: str, device=None):
    """(world, rank) from the torchrun environment; joins the process group when world > 1."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            if device is not None:
                dist.init_process_group(backend, device_id=device)
            else:
                dist.init_process_group(backend)
    return world, rank


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over all ranks (a timing: the job ends with its slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank moves bytes_per_step per step (weak scaling)."""
    return world * bytes_per_step * steps / (ms * 1e-3) / 1e9


SEQUENTIAL = False   # --sequential: the input-order float32 sum / mean mode
SCAN = False         # --scan: the segmented scan (inclusive sum and max)


def cases_of(w: W.Workload):
    if SEQUENTIAL:
        return [("f32", "sum"), ("f32", "mean")]
    if SCAN:
        return [("f32", "sum"), ("f32", "max")]
    return [(k, op) for k, op in w.cases]


def case_bytes(w: W.Workload, kind: str, op: str) -> int:
    """Algorithmic bytes of one call: a scan reads the values and offsets and
    writes one value per row; a reduction is counted by workloads.workload_bytes."""
    if SCAN:
        n = int(next(iter(w.values.values())).shape[0])
        return 8 * n + w.offsets.nbytes
    return W.workload_bytes(w, kind, op)


def step_bytes(w: W.Workload) -> int:
    return sum(case_bytes(w, k, op) for k, op in cases_of(w))


# The reduction suite: the first workload is the headline (the largest one
# that fits one GPU, 10M x 128 float32 rows in 100,000 power-law segments);
# the others are timed in the same run and reported per config.
SUITE = ("large", "mp", "skewed", "bulk", "tiny")
CPU_CASE_BUDGET_S = 1.5      # sequential oracle seconds per case in one sample


def _prefix_for(w: W.Workload, elements: float) -> int:
    """Number of leading segments whose rows hold about `elements` values
    (at least one segment)."""
    off = w.offsets.astype(np.int64)
    rows_needed = elements / max(1, w.feat)
    s = int(np.searchsorted(off - off[0], rows_needed, side="left"))
    return max(1, min(w.num_segments, s))


def _calibrated_prefix(w: W.Workload, reduce, kind: str, op: str, budget_s: float) -> int:
    """Leading segments that one sequential oracle call covers in about
    budget_s: time a small prefix, scale by values per second."""
    s_small = _prefix_for(w, 4e6)
    sub = w.offsets[: s_small + 1]
    t0 = time.perf_counter()
    reduce(w.values[kind], sub, op)
    dt = max(time.perf_counter() - t0, 1e-6)
    elems = max(1, (int(sub[-1]) - int(sub[0])) * w.feat + s_small)
    return _prefix_for(w, elems / dt * budget_s)


def _agrees(values, off, op, got, got_arg, exp, exp_arg) -> bool:
    """The parity bar: integers, min / max values and args bit for bit;
    float sums within 1e-5 * sum|x| + 1e-6 (means: over the length, plus one
    rounding)."""
    if op in ("min", "max") and not np.array_equal(got_arg, exp_arg):
        return False
    if values.dtype == np.float32 and op in ("sum", "mean"):
        o = off.astype(np.int64)
        a = np.abs(values[int(o[0]): int(o[-1])].astype(np.float64))
        a = a.reshape(a.shape[0], -1)
        cs = np.zeros((a.shape[0] + 1, a.shape[1]))
        np.cumsum(a, axis=0, out=cs[1:])
        tol = 1e-5 * (cs[o[1:] - o[0]] - cs[o[:-1] - o[0]]) + 1e-6
        e64 = exp.astype(np.float64).reshape(tol.shape)
        if op == "mean":
            tol = tol / np.maximum(np.diff(o), 1)[:, None] + 2.0 ** -23 * np.abs(e64)
        return bool((np.abs(got.astype(np.float64).reshape(tol.shape) - e64) <= tol).all())
    return bool(np.array_equal(got.view(np.uint32), exp.view(np.uint32)))


def cpu_leg(w: W.Workload, host_outs=None, budget_s: float = CPU_CASE_BUDGET_S):
    """The CPU baseline: the oracle over a bounded prefix of the workload's
    segments, every case, timed on one core (the sequential build) and on
    all cores (the OpenMP build of the same loop).  When the GPU's outputs
    are given, the oracle's outputs on that prefix are compared with them."""
    import oracle
    cases = cases_of(w)
    seq = oracle.seg_reduce_sequential if SEQUENTIAL else oracle.seg_reduce
    k0, op0 = cases[0]
    s_take = _calibrated_prefix(w, seq, k0, op0, budget_s)
    sub = w.offsets[: s_take + 1]
    rows = int(sub[-1]) - int(sub[0])
    nbytes = sum(W.algorithmic_bytes(rows, w.feat, s_take, w.offsets.dtype.itemsize, op) for _, op in cases)
    t_seq = 0.0
    checked, agree = 0, True
    for k, op in cases:
        t0 = time.perf_counter()
        r = seq(w.values[k], sub, op)
        t_seq += time.perf_counter() - t0
        if host_outs is not None:
            exp, exp_arg = r if isinstance(r, tuple) else (r, None)
            got, got_arg = host_outs[(k, op)]
            ok = _agrees(w.values[k], sub, op, got[:s_take], None if got_arg is None else got_arg[:s_take],
                         exp, exp_arg)
            agree = agree and ok
            checked += 1
    cores, t_par, par_note = 1, None, None
    if not SEQUENTIAL:
        try:
            cores = oracle.parallel_threads()
            t_par = 0.0
            for k, op in cases:
                t0 = time.perf_counter()
                oracle.seg_reduce_parallel(w.values[k], sub, op)
                t_par += time.perf_counter() - t0
        except Exception as e:     # no OpenMP on this host: one core only
            par_note = f"all-cores build unavailable: {e}"
            cores, t_par = 1, None
    sample = (f"first {s_take:,} of {w.num_segments:,} segments ({rows:,} rows), all {len(cases)} cases"
              if s_take < w.num_segments else f"whole workload, all {len(cases)} cases")
    one = {"value": nbytes / t_seq / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": sample, "seconds": t_seq}
    if t_par is not None:
        base = {"value": nbytes / t_par / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": sample, "seconds": t_par,
                "build": "the oracle's loop with OpenMP over (segment, column) pairs", "one_core": one}
    else:
        base = dict(one)
        if par_note:
            base["note"] = par_note
    parity = None
    if host_outs is not None:
        parity = {"oracle_prefix_segments": s_take, "cases": checked, "agree": agree}
    return base, parity, s_take


def run_reference(args, w: W.Workload):
    """The reference arm: the oracle as it stands (the sequential C loop) on
    one host core, each step every case over a bounded prefix of the
    workload's segments."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    cases = cases_of(w)
    offsets = w.offsets
    if SCAN:
        def reduce(v, off, op):
            # the scan of the rows the prefix of offsets covers
            return oracle.seg_scan(v[: int(off[-1])], off, op)
    else:
        reduce = oracle.seg_reduce_sequential if SEQUENTIAL else oracle.seg_reduce
    k0, op0 = cases[0]
    s_take = _calibrated_prefix(w, reduce, k0, op0, 2.0 / len(cases))
    S = w.num_segments
    sub = offsets[: s_take + 1]
    rows = int(sub[-1]) - int(sub[0])
    sample_bytes = sum((8 * int(sub[-1]) + sub.nbytes) if SCAN else
                       W.algorithmic_bytes(rows, w.feat, s_take, offsets.dtype.itemsize, op)
                       for _, op in cases)
    for _ in range(args.warmup):
        for k, op in cases:
            reduce(w.values[k], sub, op)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for k, op in cases:
            reduce(w.values[k], sub, op)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    gbs = sample_bytes * args.steps / tot / 1e9
    sample = (f"first {s_take:,} of {S:,} segments ({rows:,} rows), all {len(cases)} cases per step"
              if s_take < S else f"whole workload, all {len(cases)} cases per step")
    return {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32/s32/f32" if w.feat == 1 else "f32",
        "data": "synthetic", "config": config_of(args, w),
        "segments_per_s": s_take * len(cases) * args.steps / tot,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


WORKLOAD_TEXT = {
    "tiny": "1,000 segments, ~7.5K rows, uint32 offsets",
    "bulk": "1,000,000 segments, geometric lengths mean 16 (~16M rows), int64 offsets",
    "mp": "1,000,000 rows x 64 float32 into 10,000 segments, int64 indptr",
    "skewed": "64M float32 rows, 1M segments, Zipf(1.5) + 4 giants > 5M, 20% empty",
    "large": "10M rows x 128 float32, 100,000 power-law segments, int64 indptr",
    "large_1m": "1M rows x 128 float32, 10,000 power-law segments (a tenth of large, for profiling)",
}


def config_of(args, w):
    return {"workload": f"{w.name}: " + WORKLOAD_TEXT[w.name]
            + ("; input-order float32 mode (seg_reduce_sequential)" if SEQUENTIAL else "")
            + ("; segmented scan (seg_scan), inclusive" if SCAN else ""),
            "segments": w.num_segments, "rows": w.num_rows, "features": w.feat,
            "cases": [f"{k}:{op}" for k, op in cases_of(w)],
            "l2": "flushed before every timed call (a 2 x L2 write, then two 2 x L2 reads: clean lines, write-backs drained), outside the events"}


def kernel_of(w: W.Workload) -> str:
    if SCAN:
        return "segred::rs_scan_kernel + rs_fix_kernel (with the bitmap launches)"
    if SEQUENTIAL:
        return "segred::seg_seq_kernel"
    return "segred::seg_scalar_kernel" if w.feat == 1 else "segred::seg_rows2_kernel"


def _to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(dev).view(torch.uint32)
    return torch.from_numpy(a).to(dev)


def _host(t):
    import torch
    if t is None:
        return None
    if t.dtype == torch.uint32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    return t.cpu().numpy()


def measure_config(args, w: W.Workload, dev, world: int, flush, headline: bool):
    """Everything about one workload on the GPU: upload, a 10-run bitwise
    check of every case, warm-up, the timed steps (events per call, L2
    flushed before each), then (headline only) the end-to-end step through
    host buffers, and the CPU baseline with its oracle comparison."""
    import torch

    import segmented_reduction_csr_gb300 as sr

    local = dev.index
    cases = cases_of(w)
    stream = torch.cuda.current_stream(dev)
    dvals = {k: _to_dev(v, dev) for k, v in w.values.items()}
    doff = _to_dev(w.offsets, dev)
    outs = {}
    for k, op in cases:
        shape = (w.num_segments,) if w.feat == 1 else (w.num_segments, w.feat)
        if SCAN:
            shape = (w.num_rows,)
        o = torch.empty(shape, dtype=dvals[k].dtype, device=dev)
        a = torch.empty(shape, dtype=torch.int64, device=dev) if (op in ("min", "max") and not SCAN) else None
        outs[(k, op)] = (o, a)

    def call(k, op):
        o, a = outs[(k, op)]
        if SCAN:
            sr.seg_scan(dvals[k], doff, op, out=o)
        elif SEQUENTIAL:
            sr.seg_reduce_sequential(dvals[k], doff, op, out=o)
        else:
            sr.seg_reduce(dvals[k], doff, op, out=o, out_arg=a, with_arg=a is not None)

    # ---- ten runs of every case, bitwise identical to the first -----------------
    repro = True
    host_outs = {}
    for k, op in cases:
        call(k, op)
        o, a = outs[(k, op)]
        first = (o.clone(), a.clone() if a is not None else None)
        for _ in range(9):
            call(k, op)
            same = torch.equal(o.view(torch.int32), first[0].view(torch.int32))
            if a is not None:
                same = same and torch.equal(a, first[1])
            repro = repro and bool(same)
        host_outs[(k, op)] = (_host(first[0]), _host(first[1]))
        del first
    torch.cuda.synchronize(dev)
    assert sr.device_status(stream) == 0

    for _ in range(args.warmup):
        for k, op in cases:
            flush()
            call(k, op)
    torch.cuda.synchronize(dev)

    # ---- device-resident timing --------------------------------------------------
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps * len(cases))]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    # the GPU idled while the sampler started: one untimed round first, enqueued
    # right before the timed calls, so that the first of them pays no wake-up
    for k, op in cases:
        flush()
        call(k, op)
    wall0 = time.perf_counter()
    n = 0
    for _ in range(args.steps):
        for k, op in cases:
            flush()
            ev[n][0].record(stream)
            call(k, op)
            ev[n][1].record(stream)
            n += 1
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    per_call = [s.elapsed_time(e) for s, e in ev]             # ms
    kernel_ms = max_over_ranks(sum(per_call), world, dev)
    assert sr.device_status(stream) == 0
    peak, _ = measured_peak()
    bytes_step = step_bytes(w)
    by_case = {}
    for idx, (k, op) in enumerate(cases * args.steps):
        by_case.setdefault((k, op), []).append(per_call[idx])
    breakdown = []
    for k, op in cases:
        ms = statistics.median(by_case[(k, op)])
        b = case_bytes(w, k, op)
        breakdown.append({"config": w.name, "case": f"{k}:{op}", "us_median": ms * 1e3,
                          "gbs": b / (ms * 1e-3) / 1e9, "pct_of_peak": 100.0 * b / (ms * 1e-3) / 1e9 / peak,
                          "segments_per_s": w.num_segments / (ms * 1e-3), "bytes": b})
    res = {"w": w, "per_call": per_call, "kernel_ms": kernel_ms, "clocks": clk, "wall": wall,
           "breakdown": breakdown, "bytes_step": bytes_step, "reproducible": repro,
           "value": whole_job_gbs(world, bytes_step, args.steps, kernel_ms)}

    if headline:
        res["e2e"] = _e2e(args, w, dev, world, stream, dvals, doff, outs, call, bytes_step)
    if world == 1 and not args.no_cpu_baseline and not SCAN:
        base, parity, _ = cpu_leg(w, host_outs, CPU_CASE_BUDGET_S if headline else 0.5)
        res["cpu_baseline"] = base
        res["parity"] = parity
    del dvals, doff, outs
    torch.cuda.empty_cache()
    return res


def e2e_chunks(offsets: np.ndarray, row_bytes: int) -> list:
    """Segment ranges [a, b) for the end-to-end step: about equal row counts,
    cut at segment boundaries, one chunk per 512 MB of values (at most 8)."""
    off = np.asarray(offsets, dtype=np.int64)
    S = off.size - 1
    g = int(min(8, max(1, row_bytes // (512 << 20))))
    if S <= 0 or g == 1:
        return [(0, S)]
    o0, oS = int(off[0]), int(off[S])
    cuts = {0, S}
    for k in range(1, g):
        cuts.add(int(np.searchsorted(off[:S], o0 + (oS - o0) * k // g, side="left")))
    cuts = sorted(c for c in cuts if 0 <= c <= S)
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def _e2e(args, w, dev, world, stream, dvals, doff, outs, call, bytes_step):
    """The same bytes through host buffers: every step copies its inputs up
    from pinned memory, runs the calls and copies every output back, over
    three streams.  The offsets go up first.  Each dtype's values go up in
    row chunks cut at segment boundaries (large inputs: one per 512 MB); the
    segments of a chunk are reduced through the public call as soon as its
    rows have arrived, and their outputs go back while later chunks still
    travel.  After the timed steps the outputs on the host are compared with
    the device-resident calls' (max / min bit for bit, sums within the
    parity bar)."""
    import torch

    import segmented_reduction_csr_gb300 as sr
    cases = cases_of(w)
    host_vals = {k: torch.from_numpy(np.ascontiguousarray(v.view(np.int32) if v.dtype == np.uint32 else v)).pin_memory()
                 for k, v in w.values.items()}
    host_off = torch.from_numpy(w.offsets).pin_memory()
    host_outs = {key: (torch.empty(o.shape, dtype=o.dtype if o.dtype != torch.uint32 else torch.int32).pin_memory(),
                       torch.empty(a.shape, dtype=torch.int64).pin_memory() if a is not None else None)
                 for key, (o, a) in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in host_vals.values()) + host_off.numel() * host_off.element_size()
    d2h = sum(o.numel() * o.element_size() + (a.numel() * 8 if a is not None else 0)
              for o, a in host_outs.values())
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)
    kinds = list(dict.fromkeys(k for k, _ in cases))
    chunked = not (SCAN or SEQUENTIAL)
    offs = np.asarray(w.offsets, dtype=np.int64)
    row_bytes = max(t.numel() * t.element_size() for t in host_vals.values())
    chunks = e2e_chunks(offs, row_bytes) if chunked else [(0, w.num_segments)]

    def chunk_call(k, op, a, b):
        o, ar = outs[(k, op)]
        if chunked:
            sr.seg_reduce(dvals[k], doff[a:b + 1], op, out=o[a:b], out_arg=ar[a:b] if ar is not None else None,
                          with_arg=ar is not None)
        else:
            call(k, op)

    def e2e_step():
        up.wait_stream(stream)             # the previous step no longer reads the inputs
        with torch.cuda.stream(up):
            doff.copy_(host_off, non_blocking=True)
        for k in kinds:
            dst = dvals[k].view(torch.int32) if dvals[k].dtype == torch.uint32 else dvals[k]
            for a, b in chunks:
                r0, r1 = (int(offs[a]), int(offs[b])) if chunked else (0, dst.shape[0])
                ready = torch.cuda.Event()
                with torch.cuda.stream(up):
                    if r1 > r0:
                        dst[r0:r1].copy_(host_vals[k][r0:r1], non_blocking=True)
                    ready.record(up)
                stream.wait_event(ready)
                for kk, op in cases:
                    if kk == k:
                        chunk_call(kk, op, a, b)
                done = torch.cuda.Event()
                done.record(stream)
                down.wait_event(done)
                with torch.cuda.stream(down):
                    for (kk, op), (ho, ha) in host_outs.items():
                        if kk != k:
                            continue
                        o, ar = outs[(kk, op)]
                        src = o.view(torch.int32) if o.dtype == torch.uint32 else o
                        ho[a:b].copy_(src[a:b], non_blocking=True)
                        if ha is not None:
                            ha[a:b].copy_(ar[a:b], non_blocking=True)
        stream.wait_stream(down)           # the step ends with its outputs on the host

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # the host outputs against one device-resident call of each case: max /
    # min bit for bit, float sums and means within 1e-5 * (the mean or sum
    # of |x|) + 1e-6, the parity bar (a chunk's partition differs)
    match = True
    if chunked:
        for (k, op), (ho, ha) in host_outs.items():
            call(k, op)
            o, ar = outs[(k, op)]
            got = ho.to(dev)
            ref = o.view(torch.int32) if o.dtype == torch.uint32 else o
            if op in ("min", "max") or ref.dtype != torch.float32:
                match = match and torch.equal(got.view(torch.int32), ref.view(torch.int32))
                if ha is not None:
                    match = match and torch.equal(ha.to(dev), ar)
            else:
                absr = sr.seg_reduce(dvals[k].abs(), doff, "mean" if op == "mean" else "sum")
                match = match and bool(((got - ref).abs() <= 1e-5 * absr + 1e-6).all())
        torch.cuda.synchronize(dev)
    return {"value": whole_job_gbs(world, bytes_step, args.steps, e2e_ms), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": (f"offsets up first; each dtype's values up in {len(chunks)} row chunk(s) cut at segment "
                          "boundaries, a chunk's segments reduced by the public call as soon as its rows arrive, "
                          "their outputs back while later chunks travel"),
            "outputs_match_device_calls": bool(match)}


def run_ours(args, names):
    import torch

    import segmented_reduction_csr_gb300 as sr
    from segmented_reduction_csr_gb300 import build as srbuild

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    world, rank = dist_init("nccl", dev)
    torch.cuda.set_device(dev)
    srbuild.build()
    sr.load_library()
    flush = L2Flush(dev)
    peak, peak_kind = measured_peak()
    results = [measure_config(args, W.make(name), dev, world, flush, headline=(i == 0))
               for i, name in enumerate(names)]
    head = results[0]
    w = head["w"]
    cases = cases_of(w)
    achieved = head["bytes_step"] * args.steps / (sum(head["per_call"]) * 1e-3) / 1e9
    traffic = None if (SEQUENTIAL or SCAN) else profile_traffic(w.name)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["kernel_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "u32/s32/f32" if (w.feat == 1 and not SEQUENTIAL) else "f32", "data": "synthetic",
        "config": config_of(args, w),
        "pct_of_peak": 100.0 * head["value"] / world / peak, "peak_gbs": peak, "peak_kind": peak_kind,
        "pct_of_8tbs": 100.0 * head["value"] / world / 8000.0,
        "segments_per_s": world * w.num_segments * len(cases) * args.steps / (head["kernel_ms"] * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel_of(w) + " (every launch of the step)",
                     "peak_note": f"{peak_kind} HBM copy bandwidth",
                     "traffic_note": ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                                      "averaged over the step's cases" +
                                      ("; taken on the 1M x 128 case and scaled by rows to the full launch"
                                       if w.name == "large" else ""))},
        "e2e": head["e2e"],
        "gpu_launches": args.steps * len(cases),
        "clocks": head["clocks"],
        "wall_s_timed_region": head["wall"],
        "reproducible_10_runs": head["reproducible"],
        "breakdown": [b for r in results for b in r["breakdown"]],
        "configs": [{"workload": config_of(args, r["w"])["workload"],
                     "value": r["value"], "unit": "GB/s",
                     "pct_of_peak": 100.0 * r["value"] / world / peak,
                     "ms_per_step": r["kernel_ms"] / args.steps,
                     "segments_per_s": world * r["w"].num_segments * len(cases_of(r["w"])) * args.steps
                     / (r["kernel_ms"] * 1e-3),
                     "kernel": kernel_of(r["w"]),
                     "cases": [f"{k}:{op}" for k, op in cases_of(r["w"])],
                     "reproducible_10_runs": r["reproducible"],
                     "oracle_check": r.get("parity"),
                     "clocks": r["clocks"]} for r in results],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if head.get("parity") is not None:
        line["oracle_check"] = head["parity"]
    if world > 1:
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


PRODUCER_METRIC = "offsets-producer effective HBM GB/s (run-length encoding / flags to offsets; 1 GPU)"


def producer_input(args, w: W.Workload):
    if args.producer == "flags":
        return W.segment_flags(w.offsets)
    return W.segment_keys(w.offsets)


def producer_bytes(args, n: int, runs: int) -> int:
    """Algorithmic bytes: the input once, the outputs' valid prefixes, the count."""
    if args.producer == "flags":
        return n + 8 * (runs + 1) + 8
    if args.producer == "unique":
        return 4 * n + 4 * runs + 8
    return 4 * n + 16 * runs + 8 + 8


def producer_config(args, w: W.Workload, n: int, runs: int):
    what = "segment-start flags (uint8)" if args.producer == "flags" else "ordered segment keys (uint32)"
    return {"workload": f"{args.producer} over the {what} of the {w.name} workload",
            "elements": n, "runs": runs, "producer": args.producer,
            "l2": "flushed before every timed call (a 2 x L2 write, then two 2 x L2 reads: clean lines, write-backs drained), outside the events"}


def run_producer_reference(args, w: W.Workload):
    import oracle
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    x = producer_input(args, w)
    f = (lambda: oracle.flags_to_offsets(x)) if args.producer == "flags" else (lambda: oracle.rle(x))
    r = f()
    runs = len(r) - 1 if args.producer == "flags" else len(r[0])
    for _ in range(args.warmup):
        f()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        f()
    tot = time.perf_counter() - t0
    gbs = producer_bytes(args, x.shape[0], runs) * args.steps / tot / 1e9
    return {"metric": PRODUCER_METRIC, "value": gbs, "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8" if args.producer == "flags" else "u32",
            "data": "synthetic", "config": producer_config(args, w, x.shape[0], runs),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "whole input per step"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_producer_ours(args, w: W.Workload):
    import torch

    import segmented_reduction_csr_gb300 as sr
    from segmented_reduction_csr_gb300 import build as srbuild

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    world, rank = dist_init("nccl", dev)
    srbuild.build()
    sr.load_library()
    x = producer_input(args, w)
    n = x.shape[0]
    hx = torch.from_numpy(x.view(np.int32) if x.dtype == np.uint32 else x).pin_memory()
    dx = hx.to(dev)
    if x.dtype == np.uint32:
        dx = dx.view(torch.uint32)
    stream = torch.cuda.current_stream(dev)
    flags = args.producer == "flags"
    if flags:
        o, c = sr.seg_flags_to_offsets(dx)
        outs = (None, None, o)
    else:
        v, l, o, c = sr.seg_rle(dx, want_lengths=args.producer == "rle", want_offsets=args.producer == "rle")
        outs = (v, l, o)
    torch.cuda.synchronize(dev)
    runs = int(c.item())

    def call():
        if flags:
            sr.seg_flags_to_offsets(dx, offsets=outs[2], count=c)
        else:
            sr.seg_rle(dx, values=outs[0], lengths=outs[1], offsets=outs[2], count=c,
                       want_lengths=outs[1] is not None, want_offsets=outs[2] is not None)

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        flush()
        call()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    # the GPU idled while the sampler started: one untimed round first, enqueued
    # right before the timed calls, so that the first of them pays no wake-up
    flush()
    call()
    for s, e in ev:
        flush()
        s.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per_call = [s.elapsed_time(e) for s, e in ev]
    kernel_ms = max_over_ranks(sum(per_call), world, dev)
    assert sr.device_status(stream) == 0
    nbytes = producer_bytes(args, n, runs)
    value = whole_job_gbs(world, nbytes, args.steps, kernel_ms)

    # end to end: the input from pinned host memory, the call, the count and
    # the valid prefixes of the outputs back to pinned host memory
    host_outs = [torch.empty(t.numel(), dtype=torch.int32 if t.dtype == torch.uint32 else t.dtype).pin_memory()
                 if t is not None else None for t in outs]
    host_c = torch.empty(1, dtype=torch.int64).pin_memory()
    d2h = 8 + sum((runs + (1 if i == 2 else 0)) * t.element_size() for i, t in enumerate(outs) if t is not None)

    def e2e_step():
        (dx.view(torch.int32) if dx.dtype == torch.uint32 else dx).copy_(hx, non_blocking=True)
        call()
        host_c.copy_(c, non_blocking=True)
        for i, (t, ht) in enumerate(zip(outs, host_outs)):
            if t is None:
                continue
            k = runs + (1 if i == 2 else 0)
            ht[:k].copy_((t.view(torch.int32) if t.dtype == torch.uint32 else t)[:k], non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_producer_reference(argparse.Namespace(steps=1, warmup=0, gpus=1, producer=args.producer), w)["cpu_baseline"]
    peak, peak_kind = measured_peak()
    achieved = nbytes * args.steps / (sum(per_call) * 1e-3) / 1e9
    line = {
        "metric": PRODUCER_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": kernel_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8" if flags else "u32", "data": "synthetic",
        "config": producer_config(args, w, n, runs),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "segred::rle_count_kernel + segred::rle_write_kernel (both launches of a call)",
                     "peak_note": f"{peak_kind} HBM copy bandwidth"},
        "e2e": {"value": whole_job_gbs(world, nbytes, args.steps, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": int(hx.numel() * hx.element_size()), "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "us_per_call_median": statistics.median(per_call) * 1e3,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if world > 1:
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


SCATTER_METRIC = "unsorted scatter effective HBM GB/s (graph-reduce scatter_*; 1 GPU)"
SCATTER_CASES = ("sum", "mean", "max")


def scatter_bytes(n: int, feat: int, dim: int, op: str) -> int:
    """Algorithmic bytes: src and index read once, the outputs (and args) written once."""
    return n * feat * 4 + n * 8 + dim * feat * 4 + (dim * feat * 8 if op in ("min", "max") else 0)


def scatter_config(args, n, feat, dim):
    mode = ("; deterministic: stable sort by destination, then the segmented path"
            if getattr(args, "deterministic", False) else "; atomics")
    return {"workload": f"scatter {args.config}: {n:,} float32 rows x {feat} into {dim:,} outputs, "
                        "destinations uniform, unsorted (graph-reduce README 'Measured' shape)" + mode,
            "rows": n, "features": feat, "outputs": dim, "cases": [f"f32:{op}" for op in SCATTER_CASES],
            "l2": "flushed before every timed call (a 2 x L2 write, then two 2 x L2 reads: clean lines, write-backs drained), outside the events"}


def run_scatter_reference(args):
    import oracle
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    src, idx, dim = W.scatter_input(args.config)
    n, feat = src.shape
    for _ in range(args.warmup):
        oracle.scatter(src, idx, dim, "sum")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for op in SCATTER_CASES:
            oracle.scatter(src, idx, dim, op)
    tot = time.perf_counter() - t0
    nbytes = sum(scatter_bytes(n, feat, dim, op) for op in SCATTER_CASES)
    gbs = nbytes * args.steps / tot / 1e9
    return {"metric": SCATTER_METRIC, "value": gbs, "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": scatter_config(args, n, feat, dim),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "whole input, all cases per step"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_scatter_ours(args):
    import torch

    import segmented_reduction_csr_gb300 as sr
    from segmented_reduction_csr_gb300 import build as srbuild

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    world, rank = dist_init("nccl", dev)
    srbuild.build()
    sr.load_library()
    src, idx, dim = W.scatter_input(args.config)
    n, feat = src.shape
    hs, hi = torch.from_numpy(src).pin_memory(), torch.from_numpy(idx).pin_memory()
    ds, di = hs.to(dev), hi.to(dev)
    outs = {op: (torch.empty((dim, feat), dtype=torch.float32, device=dev),
                 torch.empty((dim, feat), dtype=torch.int64, device=dev) if op in ("min", "max") else None)
            for op in SCATTER_CASES}
    stream = torch.cuda.current_stream(dev)

    def call(op):
        o, a = outs[op]
        sr.scatter(ds, di, dim, op, out=o, out_arg=a, with_arg=a is not None,
                   deterministic=args.deterministic)

    flush = L2Flush(dev)
    for _ in range(args.warmup):
        for op in SCATTER_CASES:
            flush()
            call(op)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps * len(SCATTER_CASES))]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    # the GPU idled while the sampler started: one untimed round first, enqueued
    # right before the timed calls, so that the first of them pays no wake-up
    for op in SCATTER_CASES:
        flush()
        call(op)
    k = 0
    for _ in range(args.steps):
        for op in SCATTER_CASES:
            flush()
            ev[k][0].record(stream)
            call(op)
            ev[k][1].record(stream)
            k += 1
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per_call = [s.elapsed_time(e) for s, e in ev]
    kernel_ms = max_over_ranks(sum(per_call), world, dev)
    nbytes = sum(scatter_bytes(n, feat, dim, op) for op in SCATTER_CASES)
    breakdown = []
    for j, op in enumerate(SCATTER_CASES):
        ms = statistics.median(per_call[j::len(SCATTER_CASES)])
        breakdown.append({"case": f"f32:{op}", "us_median": ms * 1e3,
                          "gbs": scatter_bytes(n, feat, dim, op) / (ms * 1e-3) / 1e9})
    host_out = {op: (torch.empty((dim, feat), dtype=torch.float32).pin_memory(),
                     torch.empty((dim, feat), dtype=torch.int64).pin_memory() if outs[op][1] is not None else None)
                for op in SCATTER_CASES}

    def e2e_step():
        ds.copy_(hs, non_blocking=True)
        di.copy_(hi, non_blocking=True)
        for op in SCATTER_CASES:
            call(op)
            host_out[op][0].copy_(outs[op][0], non_blocking=True)
            if host_out[op][1] is not None:
                host_out[op][1].copy_(outs[op][1], non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    d2h = sum(o.numel() * 4 + (a.numel() * 8 if a is not None else 0) for o, a in host_out.values())
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_scatter_reference(argparse.Namespace(steps=1, warmup=0, gpus=1, config=args.config,
                                                       deterministic=args.deterministic))["cpu_baseline"]
    peak, peak_kind = measured_peak()
    achieved = nbytes * args.steps / (sum(per_call) * 1e-3) / 1e9
    line = {
        "metric": SCATTER_METRIC, "value": whole_job_gbs(world, nbytes, args.steps, kernel_ms),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": kernel_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": scatter_config(args, n, feat, dim),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": ("segred sort (histogram, scan, scatter passes), gather and seg_reduce launches"
                                if args.deterministic else
                                "segred::sc_add_kernel / sc_ext_kernel with their fill and finishing launches"),
                     "peak_note": f"{peak_kind} HBM copy bandwidth"},
        "e2e": {"value": whole_job_gbs(world, nbytes, args.steps, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": int(hs.numel() * 4 + hi.numel() * 8), "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * (2 + 3 + 3 if not args.deterministic else
                                      3 * (3 * ((int(dim).bit_length() + 7) // 8) + 3) + 1),
        "clocks": clk,
        "breakdown": breakdown,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if world > 1:
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default=None, choices=W.NAMES + ("mp16", "large_1m"),
                    help="one workload only (default: the suite, large first)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--producer", default=None, choices=["rle", "unique", "flags"])
    ap.add_argument("--scatter", action="store_true",
                    help="time the unsorted scatter path (sum, mean, max) on the mp or mp16 shape")
    ap.add_argument("--deterministic", action="store_true",
                    help="with --scatter: the sorted, bitwise reproducible scatter")
    ap.add_argument("--scan", action="store_true",
                    help="time the segmented scan (inclusive float32 sum and max) instead")
    ap.add_argument("--sequential", action="store_true",
                    help="time the input-order float32 sum / mean mode instead")
    args = ap.parse_args()
    global SEQUENTIAL, SCAN
    SEQUENTIAL = args.sequential
    SCAN = args.scan
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.scatter:
        args.config = args.config or "mp"
        if args.config not in ("mp", "mp16"):
            ap.error("--scatter runs on the mp or mp16 shape")
        line = run_scatter_reference(args) if args.impl == "reference" else run_scatter_ours(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.producer is not None:
        args.config = args.config or "bulk"
        if args.config not in ("bulk", "skewed"):
            ap.error("--producer runs on the bulk or skewed workload")
        w = W.make(args.config, with_values=False)
        line = run_producer_reference(args, w) if args.impl == "reference" else run_producer_ours(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.config is not None:
        names = (args.config,)
    elif SCAN or SEQUENTIAL:
        names = ("bulk",)
    else:
        names = SUITE
    if args.config == "mp16":
        ap.error("mp16 is a scatter shape")
    if args.impl == "reference":
        line = run_reference(args, W.make(names[0]))
    else:
        line = run_ours(args, names)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
