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
