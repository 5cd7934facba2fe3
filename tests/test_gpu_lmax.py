"""Ladders of other degrees (lmax = 1..5, an extension of the pages' lmax = 3
operator with the same definitions) on the GPU, against the oracle."""
import os

import numpy as np
import pytest
import torch

from equivariant_interatomic_potential_gb300 import autograd as ag
from equivariant_interatomic_potential_gb300 import workloads, zs
from gpu_helpers import assert_close, check_backward, check_csr, check_forward, dev, run_gpu

import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lmax", [1, 2, 4, 5])
@pytest.mark.parametrize("C", [32, 40, 7])
def test_ladder_matches_oracle(lmax, C):
    w = workloads.make_random(300, 20000, C, seed=10 * lmax + C, hot_node=7, hot_fraction=0.3, lmax=lmax)
    res = run_gpu(w)
    D = (lmax + 1) ** 2
    assert res["out"].shape == (300, D, C)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


@pytest.mark.parametrize("lmax", [1, 2, 4, 5])
def test_ladder_full_size_n4096(lmax):
    # the benchmarked shapes: the 4096-node, 647170-edge graph at C = 32, so the
    # kernels' rings, windows and CTA combines run exactly as timed
    w = workloads.make_workload("n4096", lmax=lmax)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        check_forward(w, res, row_ptr, perm)
        check_backward(w, res)
    finally:
        oracle.set_threads(1)


@pytest.mark.parametrize("lmax", [1, 5])
def test_ladder_deterministic_and_bad_dst(lmax):
    w = workloads.make_random(50, 8000, 32, seed=lmax, lmax=lmax)
    w.dst[::97] = -1
    w.dst[1::89] = w.N + 3
    a = run_gpu(w)
    b = run_gpu(w)
    for k in ("out", "d_coup", "d_rad", "csr_d_coup", "csr_d_rad"):
        assert np.array_equal(a[k], b[k]), k
    row_ptr, perm = check_csr(w, a)
    check_forward(w, a, row_ptr, perm)
    check_backward(w, a)
    bad = (w.dst < 0) | (w.dst >= w.N)
    assert np.all(a["d_coup"][bad] == 0) and np.all(a["d_rad"][bad] == 0)


def test_ladder_noalloc_matches_workspace_forward():
    w = workloads.make_random(200, 30000, 32, seed=3, lmax=5)
    coup, rad, dst = dev(w.coup), dev(w.rad), dev(w.dst)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    a = zs.zs_forward(coup, rad, row_ptr, perm, w.N)
    b = torch.full_like(a, float("nan"))
    zs.zs_forward_noalloc(coup, rad, row_ptr, perm, w.N, out=b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("lmax", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("C", [32, 16])
def test_ladder_autograd(lmax, C):
    # the operator's backward takes the CSR-order entry point at lmax 2, 4, 5
    # (C = 32) and the edge-order one otherwise: both against the oracle
    w = workloads.make_random(90, 12000, C, seed=8 + lmax, hot_node=4, hot_fraction=0.4, lmax=lmax)
    coup = dev(w.coup).requires_grad_(True)
    rad = dev(w.rad).requires_grad_(True)
    out = ag.zonal_scatter_from_dst(coup, rad, dev(w.dst), w.N)
    assert out.shape == (90, (lmax + 1) ** 2, C)
    d_coup, d_rad = torch.autograd.grad(out, (coup, rad), dev(w.grad_out))
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    assert_close(d_coup.cpu().numpy(), dc, adc, "d_coup")
    assert_close(d_rad.cpu().numpy(), dr, adr, "d_rad")


@pytest.mark.parametrize("lmax", [1, 2, 3, 4, 5])
def test_forward_stays_inside_its_workspace(lmax):
    # the workspace query's size is enough for every plan, and nothing is written past it
    for E in (1, 100, 5000, 20000, 300000):
        w = workloads.make_random(50, E, 32, seed=E + lmax, lmax=lmax)
        need = zs.zs_forward_workspace_bytes(E, 50, 32, lmax)
        buf = torch.full((need + 8192,), 0xAB, dtype=torch.uint8, device="cuda")
        coup, rad, dst = dev(w.coup), dev(w.rad), dev(w.dst)
        row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
        out = zs.zs_forward(coup, rad, row_ptr, perm, w.N, workspace=buf[:need])
        torch.cuda.synchronize()
        assert torch.all(buf[need:] == 0xAB), (lmax, E)
        rp, pm, _ = oracle.build_csr(w.dst, w.N)
        ref, absum = oracle.forward(w.coup, w.rad, rp, pm, w.N)
        assert_close(out.cpu().numpy(), ref, absum, f"forward lmax {lmax} E {E}")
