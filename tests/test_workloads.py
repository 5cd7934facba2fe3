"""The seeded generators produce graphs of the stated shape (no GPU)."""
import numpy as np
import pytest

from equivariant_interatomic_potential_gb300 import workloads


@pytest.mark.parametrize("name", ["tiny", "n1000", "n4096", "zipf"])
def test_config_shapes(name):
    w = workloads.make_workload(name)
    cfg = workloads.CONFIGS[name]
    assert (w.N, w.E, w.C) == (cfg["N"], cfg["E"], 32)
    assert w.dst.dtype == np.int32 and w.dst.shape == (w.E,)
    assert w.coup.shape == (w.E, 15) and w.coup.dtype == np.float32
    assert w.rad.shape == (w.E, 3, 32) and w.rad.dtype == np.float32
    assert w.grad_out.shape == (w.N, 16, 32) and w.grad_out.dtype == np.float32
    assert np.all(np.diff(w.src) >= 0)
    assert np.all(w.src != w.dst)
    assert w.dst.min() >= 0 and w.dst.max() < w.N
    assert np.all(np.abs(w.coup) <= 1.0)


def test_deterministic():
    a = workloads.make_workload("tiny")
    b = workloads.make_workload("tiny")
    for x, y in ((a.dst, b.dst), (a.coup, b.coup), (a.rad, b.rad), (a.grad_out, b.grad_out)):
        assert np.array_equal(x, y)


def test_tiny_fixed_degree():
    w = workloads.make_workload("tiny")
    assert np.array_equal(np.bincount(w.src, minlength=64), np.full(64, 32))


def test_poisson_rescale_exact():
    rng = np.random.default_rng(0)
    d = workloads.poisson_degrees(rng, 4096, 647170)
    assert d.sum() == 647170 and d.min() > 0
    assert abs(d.mean() - 647170 / 4096) < 1e-9


def test_zipf_skew():
    w = workloads.make_workload("zipf")
    indeg = np.bincount(w.dst, minlength=w.N)
    mean = w.E / w.N
    assert (indeg == 0).sum() == 205
    assert (indeg > 8 * mean).sum() >= 20
    assert indeg.max() > 100 * mean


def test_uniform_no_self_loops_small():
    rng = np.random.default_rng(3)
    src = np.repeat(np.arange(5, dtype=np.int32), 1000)
    dst = workloads.uniform_dst(rng, src, 5)
    assert np.all(dst != src)
    assert set(np.unique(dst)) == set(range(5))
