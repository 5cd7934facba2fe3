"""The degree-normalised operator (per-node factor fused into the forward,
its gradient in the backward) on the GPU, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from equivariant_interatomic_potential_gb300 import autograd as ag
from equivariant_interatomic_potential_gb300 import workloads, zs
from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu


def _factor(w, seed):
    rng = np.random.default_rng(seed)
    s = (1.0 / np.sqrt(np.maximum(np.bincount(np.clip(w.dst, 0, w.N - 1), minlength=w.N), 1))).astype(np.float32)
    s[::7] = rng.uniform(-2, 2, s[::7].shape).astype(np.float32)
    s[3] = 0.0
    return s


def _run(w, s):
    coup, rad, dst, g = dev(w.coup), dev(w.rad), dev(w.dst), dev(w.grad_out)
    s_d = dev(s)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    out, raw = zs.zs_forward_scaled(coup, rad, row_ptr, perm, s_d, w.N)
    plain = zs.zs_forward(coup, rad, row_ptr, perm, w.N)
    dc, dr, ds = zs.zs_backward_scaled(g, coup, rad, dst, s_d, w.N, out_raw=raw)
    pdc, pdr = zs.zs_backward(g, coup, rad, dst, w.N)
    torch.cuda.synchronize()
    zs.zs_check_timeouts()
    return {k: v.cpu().numpy() for k, v in dict(out=out, raw=raw, plain=plain, dc=dc, dr=dr, ds=ds,
                                                 pdc=pdc, pdr=pdr).items()}


@pytest.mark.parametrize("case", ["c32", "c40", "lmax2", "hot", "n4096", "lmax1c32", "lmax2c32", "lmax5c32"])
def test_scaled_matches_oracle(case):
    if case == "n4096":
        w = workloads.make_workload("n4096")
    else:
        # the C = 32 ladders take their own lane layouts (edge quads at lmax 1,
        # lane = channel with piece-copied rows at lmax 2, wide couplings at 5);
        # a hot node makes partials cross many CTAs
        N, E, C, lmax, hot = {"c32": (500, 40000, 32, 3, None), "c40": (200, 9000, 40, 3, None),
                              "lmax2": (150, 7000, 16, 2, None), "hot": (80, 150000, 32, 3, 9),
                              "lmax1c32": (300, 30000, 32, 1, 7), "lmax2c32": (300, 30000, 32, 2, 7),
                              "lmax5c32": (300, 30000, 32, 5, 7)}[case]
        w = workloads.make_random(N, E, C, seed=E + C, lmax=lmax, hot_node=hot, hot_fraction=0.6 if hot else 0.0)
    s = _factor(w, len(case))
    r = _run(w, s)
    row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
    out, absum, raw, absum_raw = oracle.forward_scaled(w.coup, w.rad, row_ptr, perm, w.N, s)
    assert_close(r["out"], out, absum, "scaled out")
    assert_close(r["raw"], raw, absum_raw, "out_raw")
    # fused: the plain forward's value times the factor, rounded once
    has = np.diff(row_ptr) > 0
    assert np.array_equal(r["raw"], r["plain"])
    assert np.array_equal(r["out"][has], r["plain"][has] * s[has, None, None])
    assert np.all(r["out"][~has] == 0)
    dc, dr, ds, adc, adr, ads = oracle.backward_scaled(w.grad_out, w.coup, w.rad, w.dst, w.N, s, raw)
    assert_close(r["dc"], dc, adc, "d_coup")
    assert_close(r["dr"], dr, adr, "d_rad")
    assert_close(r["ds"], ds, ads, "d_scale")
    # the edge gradients are the plain ones times the destination's factor, rounded once
    se = s[w.dst]
    assert np.array_equal(r["dc"], r["pdc"] * se[:, None])
    assert np.array_equal(r["dr"], r["pdr"] * se[:, None, None])


def test_scaled_autograd_and_determinism():
    w = workloads.make_random(300, 30000, 32, seed=77, hot_node=1, hot_fraction=0.4)
    s = _factor(w, 5)
    res = []
    for _ in range(2):
        coup = dev(w.coup).requires_grad_(True)
        rad = dev(w.rad).requires_grad_(True)
        s_d = dev(s).requires_grad_(True)
        out = ag.degree_normalised_scatter(coup, rad, dev(w.dst), s_d, w.N)
        grads = torch.autograd.grad(out, (coup, rad, s_d), dev(w.grad_out))
        res.append([out.detach().cpu().numpy()] + [x.cpu().numpy() for x in grads])
    for a, b in zip(*res):
        assert np.array_equal(a, b)
    row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
    _, _, raw, _ = oracle.forward_scaled(w.coup, w.rad, row_ptr, perm, w.N, s)
    dc, dr, ds, adc, adr, ads = oracle.backward_scaled(w.grad_out, w.coup, w.rad, w.dst, w.N, s, raw)
    assert_close(res[0][1], dc, adc, "d_coup")
    assert_close(res[0][2], dr, adr, "d_rad")
    assert_close(res[0][3], ds, ads, "d_scale")


def test_scaled_argument_checks():
    w = workloads.make_random(10, 100, 32, seed=1)
    coup, rad, dst = dev(w.coup), dev(w.rad), dev(w.dst)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    lib = zs.load()
    out = torch.empty((10, 16, 32), device="cuda")
    ws = torch.empty(zs.zs_forward_workspace_bytes(100, 10, 32), dtype=torch.uint8, device="cuda")
    st = lib.zs_forward_scaled(coup.data_ptr(), rad.data_ptr(), row_ptr.data_ptr(), perm.data_ptr(), None,
                               100, 10, 32, 3, out.data_ptr(), None, ws.data_ptr(), ws.numel(), None)
    assert st == 1 and b"node_scale" in lib.zs_last_error()
    g = dev(w.grad_out)
    s = torch.ones(10, device="cuda")
    d_scale = torch.empty(10, device="cuda")
    dcp = torch.empty((100, 15), device="cuda")
    drp = torch.empty((100, 3, 32), device="cuda")
    st = lib.zs_backward_scaled(g.data_ptr(), coup.data_ptr(), rad.data_ptr(), dst.data_ptr(), s.data_ptr(), None,
                                100, 10, 32, 3, dcp.data_ptr(), drp.data_ptr(), d_scale.data_ptr(), None)
    assert st == 1 and b"out_raw" in lib.zs_last_error()
