"""GPU parity of the offsets producers (run-length encoding, unique, flags to
offsets) against the CPU oracle, through the library's C ABI.

These are index and integer results: the bar is bit-exact equality of the
run count, values, lengths and offsets.  Outputs past the count must be left
as they were (only the prefix the count names is written)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.gpu_helpers import to_dev, to_host

pytestmark = pytest.mark.gpu

TILE = 4096          # elements per tile of the kernels (runs crossing tiles and CTAs matter)


@pytest.fixture(scope="module")
def sr():
    import segmented_reduction_csr_gb300 as m
    m.load_library()
    return m


@pytest.fixture(scope="module")
def rle_lib():
    oracle.build()
    return None          # the oracle's default library


def _check_rle(sr, rle_lib, keys, where=""):
    import torch
    n = keys.shape[0]
    ev, el, eo = oracle.rle(keys, lib=rle_lib)
    dk = to_dev(keys)
    sentinel = 0xA5A5A5A5
    dv = torch.full((n + 8,), -1, dtype=torch.int32, device="cuda").view(torch.uint32)
    dl = torch.full((n + 8,), -1, dtype=torch.int32, device="cuda").view(torch.uint32)
    do = torch.full((n + 9,), -7, dtype=torch.int64, device="cuda")
    dv.view(torch.int32).fill_(sentinel - (1 << 32))
    v, l, o, c = sr.seg_rle(dk, values=dv, lengths=dl, offsets=do)
    cnt = int(c.item())
    assert cnt == len(ev), f"{where}: count {cnt} != {len(ev)}"
    hv, hl, ho = to_host(v), to_host(l), to_host(o)
    np.testing.assert_array_equal(hv[:cnt], ev, err_msg=f"{where}: values")
    np.testing.assert_array_equal(hl[:cnt], el, err_msg=f"{where}: lengths")
    np.testing.assert_array_equal(ho[:cnt + 1], eo, err_msg=f"{where}: offsets")
    # nothing past the prefix the count names
    assert (hv[cnt:] == np.uint32(sentinel)).all(), where
    assert (hl[cnt:] == np.uint32(0xFFFFFFFF)).all(), where
    assert (ho[cnt + 1:] == -7).all(), where


SIZES = [0, 1, 2, 15, 16, 17, 255, 4095, 4096, 4097, 3 * TILE + 5, 100_003, 1_000_003]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("mean_run", [1.0, 3.0, 60.0, 5000.0])
def test_rle_random_runs(sr, rle_lib, n, mean_run):
    keys = W.random_runs(n, mean_run, seed=1000 + n % 97 + int(mean_run), distinct=1 << 32)
    _check_rle(sr, rle_lib, keys, f"n={n} mean_run={mean_run}")


@pytest.mark.parametrize("distinct", [2, 3])
def test_rle_few_distinct_keys_merge_runs(sr, rle_lib, distinct):
    keys = W.random_runs(300_001, 2.0, seed=77 + distinct, distinct=distinct)
    _check_rle(sr, rle_lib, keys, f"distinct={distinct}")


@pytest.mark.parametrize("n", [1, 4096, 1_000_000, 5_000_001])
def test_rle_all_equal_is_one_run_across_every_cta(sr, rle_lib, n):
    keys = np.full(n, 0xFFFFFFFF, dtype=np.uint32)
    _check_rle(sr, rle_lib, keys, f"all equal n={n}")


def test_rle_all_distinct(sr, rle_lib):
    keys = np.arange(1_000_003, dtype=np.uint32)[::-1].copy()
    _check_rle(sr, rle_lib, keys, "all distinct")


def test_rle_extreme_values_compare_as_uint32(sr, rle_lib):
    rng = np.random.Generator(np.random.PCG64(5))
    keys = rng.choice(np.array([0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF], np.uint32), 50_000)
    keys = np.repeat(keys, rng.integers(1, 5, size=keys.shape[0]))
    _check_rle(sr, rle_lib, keys, "extremes")


def test_rle_one_run_per_tile_boundary(sr, rle_lib):
    # a new run exactly at every tile start, and one just before / after it
    n = 40 * TILE
    keys = np.zeros(n, np.uint32)
    for t in range(1, 40):
        keys[t * TILE + (t % 3) - 1:] += 1
    _check_rle(sr, rle_lib, keys, "tile boundaries")


@pytest.mark.parametrize("shift", [1, 2, 3])
def test_rle_misaligned_keys(sr, rle_lib, shift):
    # keys that start 4, 8 or 12 bytes past a 16-byte boundary take the scalar loads
    import torch
    keys = W.random_runs(200_000, 4.0, seed=31 + shift)
    base = to_dev(np.concatenate([np.zeros(shift, np.uint32), keys]))
    dk = base[shift:]
    assert dk.data_ptr() % 16 != 0
    ev, el, eo = oracle.rle(keys, lib=rle_lib)
    v, l, o, c = sr.seg_rle(dk)
    cnt = int(c.item())
    assert cnt == len(ev)
    np.testing.assert_array_equal(to_host(v)[:cnt], ev)
    np.testing.assert_array_equal(to_host(l)[:cnt], el)
    np.testing.assert_array_equal(to_host(o)[:cnt + 1], eo)
    del torch


def test_rle_int32_keys_use_their_bits(sr, rle_lib):
    import torch
    keys = W.random_runs(100_000, 3.0, seed=8)
    ev, el, eo = oracle.rle(keys, lib=rle_lib)
    dk = torch.from_numpy(keys.view(np.int32)).cuda()
    v, l, o = sr.rle(dk)
    assert v.dtype == torch.int32
    np.testing.assert_array_equal(v.cpu().numpy().view(np.uint32), ev)
    np.testing.assert_array_equal(to_host(l), el)
    np.testing.assert_array_equal(o.cpu().numpy(), eo)


def test_unique_writes_only_values(sr, rle_lib):
    keys = W.random_runs(500_000, 7.0, seed=9)
    ev, _, _ = oracle.rle(keys, lib=rle_lib)
    v, l, o, c = sr.seg_rle(to_dev(keys), want_lengths=False, want_offsets=False)
    assert l is None and o is None
    np.testing.assert_array_equal(to_host(v)[:int(c.item())], ev)
    np.testing.assert_array_equal(to_host(sr.unique(to_dev(keys))), ev)


def test_rle_repeated_calls_identical(sr, rle_lib):
    keys = W.random_runs(2_000_000, 5.0, seed=10)
    first = [to_host(t) for t in sr.rle(to_dev(keys))]
    for _ in range(3):
        again = [to_host(t) for t in sr.rle(to_dev(keys))]
        for a, b in zip(first, again):
            np.testing.assert_array_equal(a, b)
    # no tile's look-back ran out of time
    assert sr.device_status() == 0


@pytest.mark.parametrize("name", ["bulk", "skewed"])
def test_rle_of_segment_keys_gives_back_the_offsets(sr, rle_lib, name):
    """Full-size composition: the segment id of every row of a workload, run-
    length encoded, gives the offsets of its non-empty segments; reducing over
    those offsets gives that workload's non-empty results bit for bit."""
    w = W.make(name, with_values=False)
    off = w.offsets.astype(np.int64)
    keys = W.segment_keys(off)
    _check_rle(sr, rle_lib, keys, name)
    v, l, o = sr.rle(to_dev(keys))
    nonempty = np.flatnonzero(np.diff(off) > 0)
    np.testing.assert_array_equal(to_host(v), nonempty.astype(np.uint32))
    np.testing.assert_array_equal(to_host(o), np.append(off[nonempty], off[-1]))
    if name == "bulk":
        # every bulk segment is non-empty, so the offsets come back unchanged
        import torch
        vals = W._fill_values((int(off[-1]),), 4242, "normal").astype(np.float32)
        dv = to_dev(vals)
        a = sr.seg_reduce(dv, to_dev(off), "sum")
        b = sr.seg_reduce(dv, o, "sum")
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


# ---- flags to offsets ---------------------------------------------------------------

def _check_flags(sr, rle_lib, flags, dflags=None, where=""):
    import torch
    n = flags.shape[0]
    eo = oracle.flags_to_offsets(flags, lib=rle_lib)
    df = to_dev(flags) if dflags is None else dflags
    do = torch.full((n + 5,), -3, dtype=torch.int64, device="cuda")
    o, c = sr.seg_flags_to_offsets(df, offsets=do)
    cnt = int(c.item())
    assert cnt == len(eo) - 1, f"{where}: count"
    ho = o.cpu().numpy()
    np.testing.assert_array_equal(ho[:cnt + 1], eo, err_msg=where)
    assert (ho[cnt + 1:] == -3).all(), where


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("p", [0.0, 0.001, 0.06, 0.5, 1.0])
def test_flags_random(sr, rle_lib, n, p):
    flags = W.random_flags(n, p, seed=2000 + n % 89 + int(p * 1000))
    _check_flags(sr, rle_lib, flags, where=f"n={n} p={p}")


@pytest.mark.parametrize("shift", [1, 5, 15])
def test_flags_misaligned(sr, rle_lib, shift):
    flags = W.random_flags(300_000, 0.05, seed=40 + shift)
    base = to_dev(np.concatenate([np.zeros(shift, np.uint8), flags]))
    _check_flags(sr, rle_lib, flags, dflags=base[shift:], where=f"shift={shift}")


def test_flags_bool_tensor(sr, rle_lib):
    import torch
    flags = W.random_flags(123_457, 0.1, seed=50)
    o = sr.flags_to_offsets(torch.from_numpy(flags != 0).cuda())
    np.testing.assert_array_equal(o.cpu().numpy(), oracle.flags_to_offsets(flags, lib=rle_lib))


@pytest.mark.parametrize("name", ["bulk", "skewed"])
def test_flags_of_segment_starts_give_back_the_offsets(sr, rle_lib, name):
    w = W.make(name, with_values=False)
    off = w.offsets.astype(np.int64)
    flags = W.segment_flags(off)
    _check_flags(sr, rle_lib, flags, where=name)
    nonempty = np.flatnonzero(np.diff(off) > 0)
    np.testing.assert_array_equal(sr.flags_to_offsets(to_dev(flags)).cpu().numpy(),
                                  np.append(off[nonempty], off[-1]))


def test_producer_argument_errors(sr):
    import torch
    keys = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        sr.seg_rle(keys.cpu())
    with pytest.raises(ValueError):
        sr.seg_rle(keys.view(torch.float32))
    with pytest.raises(ValueError):
        sr.seg_rle(keys, values=torch.empty(3, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        sr.seg_flags_to_offsets(torch.zeros(4, dtype=torch.int32, device="cuda"))
