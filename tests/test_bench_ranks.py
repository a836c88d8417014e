"""bench.py's multi-GPU path on the CPU: two ranks over gloo.

The reduction shards into independent replicas (one per GPU, no data-path
collective), so the only collectives in the job are a barrier and the max
of the ranks' timings.  These tests run that logic with world_size 2 on the
gloo backend, and the reference arm under torchrun, where rank 0 alone
prints the line and the other rank exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r = bench.dist_init("gloo")
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.0 + rank, w)     # rank r "took" 1 + r ms
    value = bench.whole_job_gbs(w, 10**9, 3, slowest)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump({"slowest": slowest, "value": value}, fh)
    dist.destroy_process_group()


def test_timing_is_the_max_over_two_gloo_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["slowest"] == 2.0
        # whole job: 2 ranks x 1e9 bytes x 3 steps in the slowest rank's 2 ms
        assert g["value"] == pytest.approx(2 * 1e9 * 3 / 2e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(5.0, 1) == 5.0
    assert bench.whole_job_gbs(1, 2 * 10**9, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_under_torchrun_prints_once():
    pytest.importorskip("torch")
    import oracle
    oracle.build()
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 2


def test_cpu_leg_compares_the_oracle_prefix_with_given_outputs():
    """The CPU-baseline leg times the oracle over a prefix of the segments and
    checks the outputs it is given on that prefix: outputs equal to the
    oracle's agree, one planted difference does not."""
    pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    import workloads as W
    w = W.make("tiny")
    outs = {}
    for k, op in w.cases:
        r = oracle.seg_reduce(w.values[k], w.offsets, op)
        outs[(k, op)] = r if isinstance(r, tuple) else (r, None)
    base, parity, s_take = bench.cpu_leg(w, outs, budget_s=0.05)
    assert parity["agree"] and parity["cases"] == len(w.cases) and s_take >= 1
    assert base["kind"] == "oracle" and base["value"] > 0 and base["cores"] >= 1
    bad = dict(outs)
    o, a = bad[("f32", "max")]
    a = a.copy()
    a[0] = a[0] + 1 if a[0] >= 0 else 0
    bad[("f32", "max")] = (o, a)
    assert not bench.cpu_leg(w, bad, budget_s=0.05)[1]["agree"]
    # float sums: within the bar agrees, far outside it does not
    o = outs[("f32", "sum")][0].copy()
    o[np.argmax(np.abs(o))] += 1.0
    bad2 = dict(outs)
    bad2[("f32", "sum")] = (o, None)
    assert not bench.cpu_leg(w, bad2, budget_s=0.05)[1]["agree"]


def test_suite_headline_is_the_largest_workload():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.SUITE[0] == "large"
    assert set(bench.SUITE) == {"tiny", "bulk", "mp", "skewed", "large"}


def test_end_to_end_chunks_cut_at_segment_boundaries():
    """The end-to-end step's row chunks: every segment in exactly one chunk,
    in order; about one chunk per 512 MB of values (at most 8); a segment
    longer than a chunk is never cut; small inputs go up in one piece."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import workloads as W
    w = W.make("large", with_values=False)
    off = w.offsets.astype(np.int64)
    ch = bench.e2e_chunks(off, 10_000_000 * 128 * 4)
    assert ch[0][0] == 0 and ch[-1][1] == off.size - 1
    assert all(a < b for a, b in ch) and all(ch[i][1] == ch[i + 1][0] for i in range(len(ch) - 1))
    assert 2 <= len(ch) <= 8
    rows = [int(off[b] - off[a]) for a, b in ch]
    assert sum(rows) == int(off[-1] - off[0])
    # the 5M-row segment sits whole in one chunk
    g = int(np.argmax(np.diff(off)))
    assert any(a <= g < b for a, b in ch)
    # evenly spread segments give about equal chunks
    even = np.arange(0, 8_000_001, 1000, dtype=np.int64)
    ch2 = bench.e2e_chunks(even, 8 * (512 << 20))
    assert len(ch2) == 8
    r2 = [int(even[b] - even[a]) for a, b in ch2]
    assert max(r2) - min(r2) <= 1000
    # below 512 MB, or with no segment, one chunk
    assert bench.e2e_chunks(even, 100 << 20) == [(0, even.size - 1)]
    assert bench.e2e_chunks(np.zeros(1, np.int64), 1 << 40) == [(0, 0)]
