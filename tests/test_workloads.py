"""The seeded workloads have the advertised structure and are reproducible."""
import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("name", ["tiny", "bulk", "mp", "skewed", "large"])
def test_offsets_structure(name):
    w = W.make(name, with_values=False)
    off = w.offsets.astype(np.int64)
    assert off[0] == 0 and (np.diff(off) >= 0).all()
    L = np.diff(off)
    st = {"tiny": (1000, np.uint32), "bulk": (1_000_000, np.int64), "mp": (10_000, np.int64),
          "skewed": (1_000_000, np.int64), "large": (100_000, np.int64)}[name]
    assert w.num_segments == st[0] and w.offsets.dtype == st[1]
    if name == "tiny":
        assert L.max() <= 16 and (L == 0).sum() >= 50
    if name == "bulk":
        assert L.min() >= 1 and 15.5 < L.mean() < 16.5
    if name == "mp":
        assert off[-1] == 1_000_000
    if name == "skewed":
        assert off[-1] == 64_000_000 and (L == 0).sum() == 200_000
        assert (L > 5_000_000).sum() == 4
    if name == "large":
        assert off[-1] == 10_000_000 and L.min() >= 1


def test_values_reproducible_and_shaped():
    a = W.make("tiny")
    b = W.make("tiny")
    for k in a.values:
        assert np.array_equal(a.values[k], b.values[k])
    assert a.values["f32"].min() >= -1 and a.values["f32"].max() < 1
    assert a.values["u32"].max() < 1 << 16
    m = W.make("mp")
    assert m.values["f32"].shape == (1_000_000, 64) and m.values["f32"].dtype == np.float32


def test_fill_reproducible():
    x = W._fill_values((3 * W._BLOCK + 5,), 99, "normal")
    y = np.concatenate([W._fill_values((3 * W._BLOCK + 5,), 99, "normal")])
    assert np.array_equal(x, y)


def test_scale_to_total():
    parts = W.scale_to_total([1, 1, 1000, 5], 100)
    assert parts.sum() == 100 and parts.min() >= 1 and parts.argmax() == 2


def test_algorithmic_bytes():
    # values + offsets + out (+ int64 args for min / max)
    assert W.algorithmic_bytes(10, 2, 3, 8, "sum") == 80 + 32 + 24
    assert W.algorithmic_bytes(10, 2, 3, 8, "max") == 80 + 32 + 24 + 48
