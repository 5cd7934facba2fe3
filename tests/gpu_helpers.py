"""Helpers shared by the GPU parity tests: run libzs on a workload and
compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from equivariant_interatomic_potential_gb300 import zs

TOL = 1e-5   # max |gpu - oracle| / sum|terms| per element, fp32 against fp64


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def run_gpu(w, *, backward=True):
    """CSR, forward and backward of a Workload on cuda:0; numpy results."""
    dst = dev(w.dst)
    coup = dev(w.coup)
    rad = dev(w.rad)
    row_ptr, perm, bad = zs.zs_build_csr(dst, w.N)
    out = zs.zs_forward(coup, rad, row_ptr, perm, w.N)
    res = dict(row_ptr=row_ptr.cpu().numpy(), perm=perm.cpu().numpy(), bad=int(bad.cpu()[0]),
               out=out.cpu().numpy())
    if backward:
        g = dev(w.grad_out)
        d_coup, d_rad = zs.zs_backward(g, coup, rad, dst, w.N)
        c_coup, c_rad = zs.zs_backward_csr(g, coup, rad, row_ptr, perm, w.N)
        res.update(d_coup=d_coup.cpu().numpy(), d_rad=d_rad.cpu().numpy(),
                   csr_d_coup=c_coup.cpu().numpy(), csr_d_rad=c_rad.cpu().numpy())
    torch.cuda.synchronize()
    zs.zs_check_timeouts()
    return res


def assert_close(got, ref, absum, what, tol=TOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN pattern differs"
    keep = ~nan_ref
    err, bad_zero = oracle.normalised_error(got[keep], ref[keep], np.asarray(absum)[keep])
    assert bad_zero == 0, f"{what}: {bad_zero} nonzero values where every term is zero"
    assert err <= tol, f"{what}: normalised error {err:.3e} > {tol:.1e}"
    return err


def check_csr(w, res):
    row_ptr, perm, bad = oracle.build_csr(w.dst, w.N)
    assert np.array_equal(res["row_ptr"], row_ptr), "row_ptr differs from the oracle"
    assert np.array_equal(res["perm"], perm), "perm differs from the oracle"
    assert res["bad"] == bad
    return row_ptr, perm


def check_forward(w, res, row_ptr, perm, nodes=None):
    out, absum = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N, nodes=nodes)
    got = res["out"] if nodes is None else res["out"][nodes]
    return assert_close(got, out, absum, "forward")


def check_backward(w, res, edges=None):
    """Both backward entry points against the oracle (on the sampled edges)."""
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N, edges=edges)
    errs = []
    for pre in ("", "csr_"):
        if pre + "d_coup" not in res:
            continue
        gdc = res[pre + "d_coup"] if edges is None else res[pre + "d_coup"][edges]
        gdr = res[pre + "d_rad"] if edges is None else res[pre + "d_rad"][edges]
        errs.append(assert_close(gdc, dc, adc, pre + "d_coup"))
        errs.append(assert_close(gdr, dr, adr, pre + "d_rad"))
    return errs
