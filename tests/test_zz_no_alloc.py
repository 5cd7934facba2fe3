"""zs_forward_noalloc, the forward for callers that cannot allocate device
memory (code where cudaMalloc or a caching allocator must not be called),
called through the C ABI and compared with zs_forward on two calls in a row.

This file is collected last on purpose: if it fails, every other test has
already run."""
import pytest
import torch

import oracle
from equivariant_interatomic_potential_gb300 import workloads, zs
from gpu_helpers import TOL, assert_close, dev

pytestmark = pytest.mark.gpu


def _call(lib, coup, rad, row_ptr, perm, N, out):
    return lib.zs_forward_noalloc(coup.data_ptr(), rad.data_ptr(), row_ptr.data_ptr(), perm.data_ptr(),
                                  coup.shape[0], N, rad.shape[2], 3, out.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("case", ["zipf", "odd40"])
def test_noalloc_forward_matches_workspace_forward(case):
    # zipf: C = 32 path with heavy nodes cut across CTA windows (partials in the
    # static scratch); odd40: the per-channel path (C = 40) with per-warp partials.
    # Both entry points run the same plan and kernels in the same order, so the
    # results must agree bit for bit; each is also checked against the oracle.
    w = workloads.make_workload("zipf") if case == "zipf" else workloads.make_random(300, 20000, 40, seed=40)
    lib = zs.load()
    dst, coup, rad = dev(w.dst), dev(w.coup), dev(w.rad)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    ref = zs.zs_forward(coup, rad, row_ptr, perm, w.N)
    torch.cuda.synchronize()
    want, absum = oracle.forward(w.coup, w.rad, row_ptr.cpu().numpy(), perm.cpu().numpy(), w.N)
    assert_close(ref.cpu().numpy(), want, absum, "workspace forward", tol=TOL)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call(lib, coup, rad, row_ptr, perm, w.N, out) == 0, lib.zs_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"no-alloc forward differs from zs_forward on call {call + 1}"
        assert_close(out.cpu().numpy(), want, absum, f"no-alloc forward, call {call + 1}", tol=TOL)
    zs.zs_check_timeouts()


def test_noalloc_rejects_calls_beyond_its_scratch():
    # C = 40 needs 120*C + 12 bytes per 256 edges: 300000 edges exceed the 4 MiB scratch
    E, N, C = 300000, 1000, 40
    lib = zs.load()
    coup = torch.zeros((E, 15), device="cuda")
    rad = torch.zeros((E, 3, C), device="cuda")
    row_ptr = torch.zeros(N + 1, dtype=torch.int32, device="cuda")
    perm = torch.zeros(E, dtype=torch.int32, device="cuda")
    out = torch.zeros((N, 16, C), device="cuda")
    assert _call(lib, coup, rad, row_ptr, perm, N, out) == 1
    assert b"scratch" in lib.zs_last_error()
