"""The torch.library operators over libzs: first-order autograd, no double
backward, fake implementations for tracing, CUDA graph replay.

CPU tests check the registration and shape propagation only (the operators
run no CPU code); GPU tests compare values with the oracle."""
import numpy as np
import pytest
import torch
from torch.fx.experimental.proxy_tensor import make_fx

import oracle
from equivariant_interatomic_potential_gb300 import autograd as ag
from equivariant_interatomic_potential_gb300 import workloads
from gpu_helpers import assert_close, dev


def test_operators_registered():
    for name in ("build_csr", "zonal_scatter", "zonal_scatter_backward"):
        assert hasattr(torch.ops.zs_gie, name)


def test_cpu_tensors_rejected():
    coup, rad = torch.zeros(3, 15), torch.zeros(3, 3, 32)
    dst = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        ag.zonal_scatter(coup, rad, dst, torch.zeros(5, dtype=torch.int32), dst, 4)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        ag.build_csr(dst, 4)


def test_fake_tracing_forward_and_backward():
    # traced with fake tensors: the fake implementations give every shape, no kernel runs
    def f(coup, rad, dst, g):
        out = ag.zonal_scatter_from_dst(coup, rad, dst, 9)
        d_coup, d_rad = torch.autograd.grad(out, (coup, rad), g)
        return out, d_coup, d_rad

    E, C = 40, 8
    coup = torch.randn(E, 15, requires_grad=True)
    rad = torch.randn(E, 3, C, requires_grad=True)
    dst = torch.randint(0, 9, (E,), dtype=torch.int32)
    g = torch.randn(9, 16, C)
    gm = make_fx(f, tracing_mode="fake")(coup, rad, dst, g)
    targets = {str(n.target) for n in gm.graph.nodes if n.op == "call_function"}
    assert any("zonal_scatter_backward" in t for t in targets)
    assert any("build_csr" in t for t in targets)
    outs = [n for n in gm.graph.nodes if n.op == "output"][0].args[0]
    shapes = [tuple(o.meta["val"].shape) for o in outs]
    assert shapes == [(9, 16, C), (E, 15), (E, 3, C)]


def _grads(w, dtype=torch.float32):
    coup = dev(w.coup).requires_grad_(True)
    rad = dev(w.rad).requires_grad_(True)
    dst = dev(w.dst)
    g = dev(w.grad_out)
    out = ag.zonal_scatter_from_dst(coup, rad, dst, w.N)
    d_coup, d_rad = torch.autograd.grad(out, (coup, rad), g)
    return out, d_coup, d_rad


@pytest.mark.gpu
@pytest.mark.parametrize("name,args", [("uniform", (300, 20000, 32)), ("odd_C", (77, 5000, 40)),
                                       ("hot", (64, 60000, 32))])
def test_autograd_matches_oracle(name, args):
    N, E, C = args
    w = workloads.make_random(N, E, C, seed=E + C, hot_node=3 if name == "hot" else None,
                              hot_fraction=0.7 if name == "hot" else 0.0)
    out, d_coup, d_rad = _grads(w)
    row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
    ref, absum = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N)
    assert_close(out.detach().cpu().numpy(), ref, absum, "forward")
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    assert_close(d_coup.cpu().numpy(), dc, adc, "d_coup")
    assert_close(d_rad.cpu().numpy(), dr, adr, "d_rad")


@pytest.mark.gpu
def test_no_double_backward():
    w = workloads.make_random(20, 500, 32, seed=4)
    coup = dev(w.coup).requires_grad_(True)
    rad = dev(w.rad).requires_grad_(True)
    out = ag.zonal_scatter_from_dst(coup, rad, dev(w.dst), w.N)
    g = dev(w.grad_out).requires_grad_(True)
    d_coup, d_rad = torch.autograd.grad(out, (coup, rad), g, create_graph=True)
    with pytest.raises(RuntimeError):
        torch.autograd.grad(d_rad.sum(), (coup, rad, g))


@pytest.mark.gpu
def test_compiled_function_matches_eager():
    w = workloads.make_random(128, 30000, 32, seed=12)

    def f(coup, rad, dst):
        return ag.zonal_scatter_from_dst(coup, rad, dst, 128)

    coup, rad, dst = dev(w.coup), dev(w.rad), dev(w.dst)
    eager = f(coup, rad, dst)
    compiled = torch.compile(f, backend="eager", fullgraph=True)(coup, rad, dst)
    assert torch.equal(eager, compiled)


@pytest.mark.gpu
@pytest.mark.parametrize("lmax", [3, 2])
def test_cuda_graph_replay_with_new_inputs(lmax):
    # the C = 32 forward combines nodes that cross CTA windows with per-launch
    # tags; replays of one captured graph must each see their own partials
    # (lmax 3: quad layout; lmax 2: lane-per-channel layout)
    N, E, C = 64, 120000, 32
    ws = [workloads.make_random(N, E, C, seed=s, hot_node=5, hot_fraction=0.6, lmax=lmax) for s in (21, 22, 23)]
    coup, rad, dst, g = (dev(ws[0].coup), dev(ws[0].rad), dev(ws[0].dst), dev(ws[0].grad_out))
    row_ptr, perm = ag.build_csr(dst, N)          # warm-up outside the capture
    ag.zonal_scatter(coup, rad, dst, row_ptr, perm, N)
    ag.zonal_scatter_backward(g, coup, rad, dst, row_ptr, perm, N)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s), torch.cuda.graph(graph, stream=s):
        rp, pm = ag.build_csr(dst, N)
        out = ag.zonal_scatter(coup, rad, dst, rp, pm, N)
        d_coup, d_rad = ag.zonal_scatter_backward(g, coup, rad, dst, rp, pm, N)
    torch.cuda.synchronize()
    for w in ws[1:] + ws[:1]:
        coup.copy_(torch.from_numpy(w.coup))
        rad.copy_(torch.from_numpy(w.rad))
        dst.copy_(torch.from_numpy(w.dst))
        g.copy_(torch.from_numpy(w.grad_out))
        graph.replay()
        torch.cuda.synchronize()
        r2, p2, _ = oracle.build_csr(w.dst, N)
        assert np.array_equal(pm.cpu().numpy(), p2)
        ref, absum = oracle.forward(w.coup, w.rad, r2, p2, N)
        assert_close(out.cpu().numpy(), ref, absum, "forward")
        dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, N)
        assert_close(d_coup.cpu().numpy(), dc, adc, "d_coup")
        assert_close(d_rad.cpu().numpy(), dr, adr, "d_rad")


def test_backward_entry_point_per_ladder():
    # the CSR-order backward where it measured faster (lmax 2, 4, 5 at C = 32)
    assert [ag.uses_csr_backward(l, 32) for l in (1, 2, 3, 4, 5)] == [False, True, False, True, True]
    assert not any(ag.uses_csr_backward(l, 40) for l in (1, 2, 3, 4, 5))


@pytest.mark.gpu
def test_operator_raises_on_timeout_flag():
    # a bounded wait that runs out sets the registered page-locked flag; the
    # next operator call raises, and the flag stays clear after normal calls
    from equivariant_interatomic_potential_gb300 import zs
    w = workloads.make_random(50, 3000, 32, seed=5)
    coup, rad, dst = dev(w.coup), dev(w.rad), dev(w.dst)
    flag = zs.timeout_flag()
    zs.zs_check_timeouts()
    flag[0] = 0
    out = ag.zonal_scatter_from_dst(coup, rad, dst, w.N)
    torch.cuda.synchronize()
    assert int(flag[0]) == 0
    lib = zs.load()
    assert lib.zs_selftest_bounded_wait(8, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(flag[0]) == 1
    with pytest.raises(zs.ZsError, match="ZS_ERR_TIMEOUT"):
        ag.zonal_scatter_from_dst(coup, rad, dst, w.N)
    assert int(flag[0]) == 0                       # the raise cleared it
    assert lib.zs_check_timeouts() == 4            # the counter saw it too
    out2 = ag.zonal_scatter_from_dst(coup, rad, dst, w.N)
    torch.cuda.synchronize()
    assert int(flag[0]) == 0 and torch.equal(out, out2)


@pytest.mark.gpu
@pytest.mark.parametrize("how", ["slots", "channels", "edges"])
def test_sliced_view_radial_inputs(how):
    # A radial operand that is a view into a wider buffer (a slice of its
    # slot axis, of its channel axis, or every other edge row).  As on the
    # pages, the operator makes its inputs contiguous before the kernels;
    # the gradient flows back into the wider buffer through the view.
    w = workloads.make_random(300, 20000, 32, seed=31, hot_node=4, hot_fraction=0.3)
    E, C = w.E, w.C
    rad = dev(w.rad)
    if how == "slots":
        base = torch.zeros((E, 4, C), device="cuda")
        base[:, 1:] = rad
        view = lambda b: b[:, 1:, :]  # noqa: E731
    elif how == "channels":
        base = torch.zeros((E, 3, C + 8), device="cuda")
        base[:, :, 4:4 + C] = rad
        view = lambda b: b[:, :, 4:4 + C]  # noqa: E731
    else:
        base = torch.zeros((2 * E, 3, C), device="cuda")
        base[::2] = rad
        view = lambda b: b[::2]  # noqa: E731
    base.requires_grad_(True)
    coup = dev(w.coup).requires_grad_(True)
    v = view(base)
    assert not v.is_contiguous()
    out = ag.zonal_scatter_from_dst(coup, v, dev(w.dst), w.N)
    d_coup, d_base = torch.autograd.grad(out, (coup, base), dev(w.grad_out))
    row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
    ref, absum = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N)
    assert_close(out.detach().cpu().numpy(), ref, absum, "forward")
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    assert_close(d_coup.cpu().numpy(), dc, adc, "d_coup")
    assert_close(view(d_base).cpu().numpy(), dr, adr, "d_rad")
    mask = torch.ones_like(d_base, dtype=torch.bool)
    view(mask).fill_(False)
    assert torch.all(d_base[mask] == 0)
