"""The paths on several streams at once: each (device, stream) keeps its own
scratch, so calls enqueued on different streams without any ordering between
them must not disturb one another.  Results are checked against the oracles
after one synchronisation."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_helpers import assert_parity, to_dev, to_host

pytestmark = pytest.mark.gpu


def test_scan_rle_scatter_and_reduce_on_four_streams():
    import torch
    import segmented_reduction_csr_gb300 as sr
    rng = np.random.default_rng(123)
    n = 2_000_003
    vals = rng.standard_normal(n).astype(np.float32)
    off = W.random_offsets(rng, n, 50_000, empty_frac=0.1)
    keys = W.random_runs(n, 5.0, seed=124)
    rows = rng.standard_normal((300_000, 16)).astype(np.float32)
    idx = rng.integers(0, 1000, size=300_000).astype(np.int64)
    dv, do, dk, dr, di = to_dev(vals), to_dev(off), to_dev(keys), to_dev(rows), to_dev(idx)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    results = {}
    for rep in range(3):
        with torch.cuda.stream(streams[0]):
            results["scan"] = sr.seg_scan(dv, do, "max")
        with torch.cuda.stream(streams[1]):
            results["rle"] = sr.seg_rle(dk)
        with torch.cuda.stream(streams[2]):
            results["scatter"] = sr.scatter(dr, di, 1000, "max", deterministic=True)
        with torch.cuda.stream(streams[3]):
            results["reduce"] = sr.seg_reduce(dv, do, "min")
    torch.cuda.synchronize()
    assert (to_host(results["scan"]).view(np.uint32) == oracle.seg_scan(vals, off, "max").view(np.uint32)).all()
    v, l, o, c = results["rle"]
    ev, el, eo = oracle.rle(keys)
    cnt = int(c.item())
    assert cnt == len(ev)
    assert (to_host(v)[:cnt] == ev).all() and (to_host(l)[:cnt] == el).all() and (to_host(o)[:cnt + 1] == eo).all()
    go, ga = results["scatter"]
    eo2, ea2 = oracle.scatter(rows, idx, 1000, "max")
    assert (to_host(go) == eo2).all() and (to_host(ga) == ea2).all()
    ro, ra = results["reduce"]
    assert_parity(vals, off, "min", to_host(ro), to_host(ra), where="reduce on stream 3")
    assert sr.device_status() == 0
