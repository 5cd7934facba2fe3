"""bench.py's byte model and reporting helpers, on CPU.

The algorithmic bytes are what each step must move at least: every edge's
index, coupling row and radial row once (and, for the backward, their two
gradients once), the node rows once.  Pinned here to sums worked out by hand
for the n4096 graph at the pages' shapes (lmax 3: 15 coupling rows, 3 radial
slots, 16 node rows, C = 32)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

N, E, C = 4096, 647170, 32


def test_bytes_n4096_by_hand():
    b = bench.algorithmic_bytes(N, E, C)
    # forward: perm 4 + coup 15*4 + rad 3*32*4 = 448 B per edge; row_ptr; out 16*32*4 B per node
    assert b["fwd"] == E * 448 + 4 * (N + 1) + N * 2048 == 298_337_156
    # backward: dst 4 + coup 60 + rad 384 + d_coup 60 + d_rad 384 = 892 B per edge; g read once
    assert b["bwd"] == E * 892 + N * 2048 == 585_664_248
    # CSR: dst read and perm written, 8 B per edge, plus row_ptr
    assert b["csr"] == E * 8 + 4 * (N + 1) == 5_193_748


def test_bytes_other_ladders():
    # lmax 1: 3 coupling rows, 1 radial slot, 4 node rows; lmax 5: 35, 5, 36
    for lmax, R, D in ((1, 3, 4), (2, 8, 9), (4, 24, 25), (5, 35, 36)):
        b = bench.algorithmic_bytes(N, E, C, lmax)
        assert b["fwd"] == E * (4 + 4 * R + 128 * lmax) + 4 * (N + 1) + N * D * 128
        assert b["bwd"] == E * (4 + 8 * R + 256 * lmax) + N * D * 128
        assert b["csr"] == E * 8 + 4 * (N + 1)


def test_scaled_extra_bytes():
    # the factor (4 B per node) and the unscaled output: written by the
    # forward, read again with g by the backward, which also writes d_scale
    x = bench.scaled_extra_bytes(N, C, 3)
    assert x["fwd"] == 4 * N + 2048 * N
    assert x["bwd"] == 4 * N + 2 * 2048 * N + 4 * N


def test_metric_names():
    assert bench.metric_for(3) == bench.METRIC
    assert "lmax=2" in bench.metric_for(2)
    assert bench.metric_for(3, scaled=True).startswith("degree-normalised")


def test_job_throughput_counts_all_ranks():
    # units of every rank over the slowest rank's time
    assert bench.job_throughput(1000, 10, 2.0, 4) == 1000 * 10 * 4 / 2e-3


def test_kernel_figures():
    # 1 GB in 200 us is 5000 GB/s: 0.5 of a 10000 GB/s peak, 0.625 of 8000
    ab = {"fwd": 10 ** 9}
    k = bench.kernel_figures(ab, {"fwd": 200.0}, {"fwd": [250.0, 250.0, 400.0]}, 1000, 10000.0, "measured", ("fwd",))
    f = k["fwd"]
    assert abs(f["GBs"] - 5000.0) < 1e-9
    assert abs(f["frac_of_measured"] - 0.5) < 1e-12
    assert abs(f["frac_of_nominal_8000"] - 0.625) < 1e-12
    assert abs(f["edges_per_s"] - 1000 / 200e-6) < 1e-3
    assert f["us_in_step_mean"] == 300.0 and f["us_in_step_median"] == 250.0
    assert abs(f["frac_in_step"] - 10 ** 9 / 300e-6 / 1e9 / 10000.0) < 1e-12


def test_kernel_figures_marginal():
    # the marginal cost in the step: 1 GB in 250 us is 4000 GB/s, 0.4 of a 10000 GB/s peak
    ab = {"fwd": 10 ** 9, "bwd": 10 ** 9}
    k = bench.kernel_figures(ab, {"fwd": 200.0, "bwd": 200.0}, {"fwd": [300.0], "bwd": [300.0]}, 1000, 10000.0,
                             "measured", ("fwd", "bwd"), {"fwd": 250.0})
    assert k["fwd"]["us_marginal_in_step"] == 250.0
    assert abs(k["fwd"]["frac_marginal_in_step"] - 0.4) < 1e-12
    assert "us_marginal_in_step" not in k["bwd"]
