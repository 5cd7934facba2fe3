"""libzs on the GPU against the CPU oracle: CSR bit-exact, forward and
backward within 1e-5 normalised error, bitwise run-to-run determinism, edge
cases, and no writes outside the outputs."""
import os

import numpy as np
import pytest
import torch

import oracle
from equivariant_interatomic_potential_gb300 import workloads, zs
from gpu_helpers import TOL, assert_close, check_backward, check_csr, check_forward, dev, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    zs.load()
    torch.cuda.init()


# ------------------------------------------------------------------ named configurations

@pytest.mark.parametrize("name", ["tiny", "n1000", "n4096", "zipf"])
def test_config_full_parity(name):
    w = workloads.make_workload(name)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)
    deg = np.diff(row_ptr)
    assert np.all(res["out"][deg == 0] == 0)
    assert np.all(res["out"][:, 0, :] == 0)


def test_large_config_full_parity():
    # every CSR entry, every node of out and every edge of both backward entry
    # points against the oracle (its node and edge loops on all host cores;
    # the edges in chunks to bound host memory)
    w = workloads.make_workload("large")
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        check_forward(w, res, row_ptr, perm)
        deg = np.diff(row_ptr)
        assert np.all(res["out"][deg == 0] == 0) and np.all(res["out"][:, 0, :] == 0)
        chunk = 1 << 19
        for e0 in range(0, w.E, chunk):
            check_backward(w, res, edges=np.arange(e0, min(w.E, e0 + chunk), dtype=np.int64))
    finally:
        oracle.set_threads(1)


# ------------------------------------------------------------------ shapes and edge cases

@pytest.mark.parametrize("C", [1, 3, 4, 8, 16, 31, 32, 33, 40, 64, 128])
def test_channel_counts(C):
    w = workloads.make_random(200, 9000, C, seed=C)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


def test_pages_odd_channel_shape():
    # E=777 edges, N=33 nodes, C=40 channels
    w = workloads.make_random(33, 777, 40, seed=777)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


@pytest.mark.parametrize("E", [1, 31, 32, 33, 37, 255, 256, 257, 2047, 2048, 2049, 8192, 8193, 16385])
def test_edge_count_boundaries(E):
    w = workloads.make_random(97, E, 32, seed=E)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


@pytest.mark.parametrize("E", [152 * 15 * 96, 152 * 15 * 96 + 1])
def test_forward_warp_count_switch(E):
    # on a 152-SM GB300 the lmax-3 forward runs 10 warps per CTA up to 218880
    # edges (15-warp windows under 96 positions) and 15 from the next edge on
    w = workloads.make_random(1000, E, 32, seed=E)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


@pytest.mark.parametrize("N,E,hot", [(1, 5000, None), (50, 20000, 7), (3000, 100000, 11), (2, 70000, 0)])
def test_heavy_nodes(N, E, hot):
    # one node takes most edges: its CSR run crosses many warp and CTA windows
    w = workloads.make_random(N, E, 32, seed=N + E, self_loops=True, hot_node=hot, hot_fraction=0.8)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


@pytest.mark.parametrize("scaled", [False, True])
def test_hot_destination_slot_is_bitwise_neutral(scaled):
    # Each edge's gradients depend on its own rows and g[dst] only.  On a graph
    # where one node takes 60 % of the edges the edge-order backward serves that
    # node's cotangent rows from a per-CTA copy; spread the same edges out
    # between 63 edges to uniformly drawn nodes each (about 1 % hot: no copy) and
    # every edge's gradients must come out bit for bit the same.
    N, E, k = 2000, 10000, 64
    w = workloads.make_random(N, E, 32, seed=41, hot_node=5, hot_fraction=0.6)
    filler = workloads.make_random(N, E * (k - 1), 32, seed=42)
    dst2 = filler.dst.reshape(E, k - 1)
    dst2 = np.concatenate([w.dst[:, None], dst2], axis=1).reshape(-1)
    coup2 = np.concatenate([w.coup[:, None], filler.coup.reshape(E, k - 1, 15)], axis=1).reshape(-1, 15)
    rad2 = np.concatenate([w.rad[:, None], filler.rad.reshape(E, k - 1, 3, 32)], axis=1).reshape(-1, 3, 32)
    g = dev(w.grad_out)
    if scaled:
        s = dev(np.random.default_rng(7).uniform(0.5, 2.0, N).astype(np.float32))
        raw = dev(np.random.default_rng(8).standard_normal((N, 16, 32)).astype(np.float32))
        a = zs.zs_backward_scaled(g, dev(w.coup), dev(w.rad), dev(w.dst), s, N, out_raw=raw)
        b = zs.zs_backward_scaled(g, dev(coup2), dev(rad2), dev(dst2), s, N, out_raw=raw)
    else:
        a = zs.zs_backward(g, dev(w.coup), dev(w.rad), dev(w.dst), N)
        b = zs.zs_backward(g, dev(coup2), dev(rad2), dev(dst2), N)
    assert torch.equal(a[0], b[0][::k]) and torch.equal(a[1], b[1][::k])
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, N)
    if not scaled:
        assert_close(a[0].cpu().numpy(), dc, adc, "d_coup")
        assert_close(a[1].cpu().numpy(), dr, adr, "d_rad")
    zs.zs_check_timeouts()


@pytest.mark.parametrize("C", [32, 5])
def test_no_edges(C):
    w = workloads.make_random(10, 0, C, seed=1)
    dst = dev(w.dst)
    row_ptr, perm, bad = zs.zs_build_csr(dst, w.N)
    assert row_ptr.cpu().numpy().tolist() == [0] * 11 and int(bad.cpu()[0]) == 0
    out = torch.full((10, 16, C), float("nan"), device="cuda")
    zs.zs_forward(dev(w.coup), dev(w.rad), row_ptr, perm, w.N, out=out)
    assert torch.all(out == 0)
    d_coup, d_rad = zs.zs_backward(dev(w.grad_out), dev(w.coup), dev(w.rad), dst, w.N)
    assert d_coup.numel() == 0 and d_rad.numel() == 0


def test_no_nodes():
    # every destination is out of range when N == 0
    w = workloads.make_random(5, 300, 32, seed=2)
    dst = dev(w.dst)
    row_ptr, perm, bad = zs.zs_build_csr(dst, 0)
    assert row_ptr.cpu().numpy().tolist() == [0]
    assert int(bad.cpu()[0]) == 300
    assert np.array_equal(perm.cpu().numpy(), np.arange(300))
    out = zs.zs_forward(dev(w.coup), dev(w.rad), row_ptr, perm, 0)
    assert out.shape == (0, 16, 32)
    d_coup, d_rad = zs.zs_backward(torch.zeros((0, 16, 32), device="cuda"), dev(w.coup), dev(w.rad), dst, 0)
    assert torch.all(d_coup == 0) and torch.all(d_rad == 0)


@pytest.mark.parametrize("C", [32, 7])
def test_out_of_range_destinations(C):
    w = workloads.make_random(300, 20000, C, seed=3)
    rng = np.random.default_rng(4)
    idx = rng.choice(w.E, 700, replace=False)
    w.dst[idx[:300]] = -1 - rng.integers(0, 5, 300)
    w.dst[idx[300:]] = w.N + rng.integers(0, 5, 400)
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    assert res["bad"] == 700
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)
    assert np.all(res["d_coup"][idx] == 0) and np.all(res["d_rad"][idx] == 0)


@pytest.mark.parametrize("N,bad_fraction", [(0, 1.0), (50, 0.8), (4096, 0.5)])
def test_out_of_range_destinations_dominate(N, bad_fraction):
    # most edges share one out-of-range destination: the edge-order backward's
    # per-CTA hot-destination vote must pass over it (it has no cotangent rows)
    w = workloads.make_random(max(N, 1), 60000, 32, seed=17 + N)
    rng = np.random.default_rng(18 + N)
    idx = rng.random(w.E) < bad_fraction
    w.dst[idx] = N + 3
    w.dst[~idx] = np.minimum(w.dst[~idx], max(N - 1, 0))
    w = workloads.Workload(w.name, N, w.E, w.C, w.seed, w.src, w.dst, w.coup, w.rad, w.grad_out[:N])
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)
    assert np.all(res["d_coup"][idx] == 0) and np.all(res["d_rad"][idx] == 0)


@pytest.mark.parametrize("N", [1, 2, 255, 256, 257, 4095, 4096, 65535, 65536, 65537, 300000])
def test_csr_radix_pass_boundaries(N):
    rng = np.random.default_rng(N)
    E = 50000
    dst = rng.integers(0, N, size=E).astype(np.int32)
    dst[:50] = N - 1
    row_ptr, perm, bad = zs.zs_build_csr(dev(dst), N)
    r2, p2, b2 = oracle.build_csr(dst, N)
    assert np.array_equal(row_ptr.cpu().numpy(), r2)
    assert np.array_equal(perm.cpu().numpy(), p2)
    assert int(bad.cpu()[0]) == b2 == 0


@pytest.mark.parametrize("E,N", [(2_000_000, 3000), (70_000, 5118), (70_000, 5119), (70_000, 5120), (513, 0), (1, 1)])
def test_csr_counting_path_limits(E, N):
    # the one-pass counting construction covers N + 1 <= 5120 (radix beyond);
    # 2M edges give tiles of 8192 edges in more than one wave
    rng = np.random.default_rng(E + N)
    dst = rng.integers(-2, N + 2, size=E).astype(np.int32)
    if N > 0:
        dst[: E // 4] = N - 1
    row_ptr, perm, bad = zs.zs_build_csr(dev(dst), N)
    r2, p2, b2 = oracle.build_csr(dst, N)
    assert np.array_equal(row_ptr.cpu().numpy(), r2)
    assert np.array_equal(perm.cpu().numpy(), p2)
    assert int(bad.cpu()[0]) == b2


def test_self_loops_and_nan():
    w = workloads.make_random(40, 6000, 32, seed=9, self_loops=True)
    e_nan = 1234
    w.rad[e_nan, 1, 5] = np.nan
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)
    n = w.dst[e_nan]
    assert np.isnan(res["out"][n, 4:9, 5]).all()
    assert np.isfinite(np.delete(res["out"], n, axis=0)).all()
    assert np.isnan(res["d_coup"][e_nan, 3:8]).all() and np.isfinite(res["d_coup"][e_nan, [0, 1, 2] + list(range(8, 15))]).all()
    assert np.isfinite(res["d_rad"]).all()


def test_misaligned_views_take_the_channel_path():
    # rad / out / g / d_rad one float off a 16-byte boundary: same results
    w = workloads.make_random(120, 7000, 32, seed=10)
    E, N = w.E, w.N
    rad_buf = torch.zeros(E * 96 + 1, device="cuda")
    rad = rad_buf[1:].view(E, 3, 32)
    rad.copy_(dev(w.rad))
    coup = dev(w.coup)
    dst = dev(w.dst)
    row_ptr, perm, _ = zs.zs_build_csr(dst, N)
    out_buf = torch.zeros(N * 512 + 1, device="cuda")
    out = zs.zs_forward(coup, rad, row_ptr, perm, N, out=out_buf[1:].view(N, 16, 32))
    g_buf = torch.zeros(N * 512 + 1, device="cuda")
    g = g_buf[1:].view(N, 16, 32)
    g.copy_(dev(w.grad_out))
    dr_buf = torch.zeros(E * 96 + 1, device="cuda")
    d_coup, d_rad = zs.zs_backward(g, coup, rad, dst, N, d_rad=dr_buf[1:].view(E, 3, 32))
    res = dict(out=out.cpu().numpy(), d_coup=d_coup.cpu().numpy(), d_rad=d_rad.cpu().numpy())
    rp, pm = oracle.build_csr(w.dst, N)[:2]
    check_forward(w, res, rp, pm)
    check_backward(w, res)


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout():
    lib = zs.load()
    zs.zs_check_timeouts()                      # nothing pending
    for spins in (1, 1000):
        assert lib.zs_selftest_bounded_wait(spins, torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert lib.zs_check_timeouts() == 4     # ZS_ERR_TIMEOUT, counter cleared
        assert b"bounded waits ran out" in lib.zs_last_error()
        assert lib.zs_check_timeouts() == 0
    zs.zs_check_timeouts()                      # the binding's flag word (if registered) is cleared too
    # the context is still usable afterwards
    w = workloads.make_workload("tiny")
    res = run_gpu(w)
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)


@pytest.mark.parametrize("where", ["device", "pinned"])
def test_timeout_flag_word(where):
    # a registered flag word is set by a wait that runs out and by nothing
    # else: the caller sees the timeout without synchronising the device
    lib = zs.load()
    stream = torch.cuda.current_stream().cuda_stream
    flag = torch.zeros(1, dtype=torch.int32, device="cuda") if where == "device" else \
        torch.zeros(1, dtype=torch.int32, pin_memory=True)
    try:
        assert lib.zs_set_timeout_flag(flag.data_ptr()) == 0, lib.zs_last_error()
        w = workloads.make_workload("n1000")
        res = run_gpu(w)                         # a normal run: flag stays clear
        assert int(flag.cpu()[0]) == 0
        assert lib.zs_selftest_bounded_wait(16, stream) == 0
        torch.cuda.synchronize()
        assert int(flag.cpu()[0]) == 1
        assert lib.zs_check_timeouts() == 4
        flag.zero_()
        torch.cuda.synchronize()
        res2 = run_gpu(w)
        assert int(flag.cpu()[0]) == 0
        assert np.array_equal(res["out"], res2["out"]) and np.array_equal(res["d_rad"], res2["d_rad"])
    finally:
        # put back the binding's own page-locked flag (or none)
        own = zs._flags.get(torch.cuda.current_device())
        assert lib.zs_set_timeout_flag(own.data_ptr() if own is not None else None) == 0


# ------------------------------------------------------------------ determinism and ownership

@pytest.mark.parametrize("name", ["n4096", "zipf", "large"])
def test_bitwise_deterministic(name):
    # large: the radix CSR and the backward's 8-warp, 3-stage ring (cotangent
    # block beyond 16 MiB)
    w = workloads.make_workload(name)
    dst, coup, rad, g = dev(w.dst), dev(w.coup), dev(w.rad), dev(w.grad_out)
    ref = None
    for _ in range(10):
        row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
        out = zs.zs_forward(coup, rad, row_ptr, perm, w.N)
        d_coup, d_rad = zs.zs_backward(g, coup, rad, dst, w.N)
        c_coup, c_rad = zs.zs_backward_csr(g, coup, rad, row_ptr, perm, w.N)
        cur = [t.clone() for t in (row_ptr, perm, out, d_coup, d_rad, c_coup, c_rad)]
        if ref is None:
            ref = cur
        else:
            for a, b in zip(ref, cur):
                assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                                   b.view(torch.int32) if b.dtype == torch.float32 else b)


@pytest.mark.parametrize("C", [32, 40])
def test_inputs_untouched_and_guard_bands(C):
    w = workloads.make_workload("zipf") if C == 32 else workloads.make_random(500, 60000, C, seed=12)
    E, N = w.E, w.N
    G = 4096
    canary = -1.75 * 2.0 ** 100   # exactly representable in fp32

    def banded(n, dtype):
        buf = torch.full((n + 2 * G,), canary, device="cuda").to(dtype) if dtype == torch.float32 else \
            torch.full((n + 2 * G,), -123456789, dtype=torch.int32, device="cuda")
        return buf, buf[G:G + n]

    dst, coup, rad, g = dev(w.dst), dev(w.coup), dev(w.rad), dev(w.grad_out)
    before = [t.clone() for t in (dst, coup, rad, g)]
    rp_buf, rp = banded(N + 1, torch.int32)
    pm_buf, pm = banded(E, torch.int32)
    bd_buf, bd = banded(1, torch.int32)
    zs.zs_build_csr(dst, N, row_ptr=rp, perm=pm, bad_dst_count=bd)
    out_buf, out = banded(N * 16 * C, torch.float32)
    zs.zs_forward(coup, rad, rp, pm, N, out=out.view(N, 16, C))
    dc_buf, dc = banded(E * 15, torch.float32)
    dr_buf, dr = banded(E * 3 * C, torch.float32)
    zs.zs_backward(g, coup, rad, dst, N, d_coup=dc.view(E, 15), d_rad=dr.view(E, 3, C))
    torch.cuda.synchronize()
    for a, b in zip(before, (dst, coup, rad, g)):
        assert torch.equal(a, b), "an input was modified"
    for buf in (rp_buf, pm_buf, bd_buf, out_buf, dc_buf, dr_buf):
        head, tail = buf[:G], buf[-G:]
        assert torch.equal(head, torch.full_like(head, head[0].item())) and torch.equal(tail, head)
    assert out_buf[0].item() == canary and rp_buf[0].item() == -123456789
    res = dict(row_ptr=rp.cpu().numpy(), perm=pm.cpu().numpy(), bad=int(bd.cpu()[0]),
               out=out.view(N, 16, C).cpu().numpy(), d_coup=dc.view(E, 15).cpu().numpy(),
               d_rad=dr.view(E, 3, C).cpu().numpy())
    row_ptr, perm = check_csr(w, res)
    check_forward(w, res, row_ptr, perm)
    check_backward(w, res)


def test_output_fully_overwritten():
    w = workloads.make_workload("zipf")
    dst, coup, rad, g = dev(w.dst), dev(w.coup), dev(w.rad), dev(w.grad_out)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    out = torch.full((w.N, 16, 32), float("nan"), device="cuda")
    zs.zs_forward(coup, rad, row_ptr, perm, w.N, out=out)
    d_coup = torch.full((w.E, 15), float("nan"), device="cuda")
    d_rad = torch.full((w.E, 3, 32), float("nan"), device="cuda")
    zs.zs_backward(g, coup, rad, dst, w.N, d_coup=d_coup, d_rad=d_rad)
    assert torch.isfinite(out).all() and torch.isfinite(d_coup).all() and torch.isfinite(d_rad).all()
    deg = torch.diff(row_ptr)
    assert torch.all(out[deg == 0] == 0)


def test_streams_are_honoured():
    w = workloads.make_workload("n1000")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dst, coup, rad, g = dev(w.dst), dev(w.coup), dev(w.rad), dev(w.grad_out)
        row_ptr, perm, _ = zs.zs_build_csr(dst, w.N, stream=s)
        out = zs.zs_forward(coup, rad, row_ptr, perm, w.N, stream=s)
        d_coup, d_rad = zs.zs_backward(g, coup, rad, dst, w.N, stream=s)
    s.synchronize()
    res = dict(row_ptr=row_ptr.cpu().numpy(), perm=perm.cpu().numpy(), bad=0, out=out.cpu().numpy(),
               d_coup=d_coup.cpu().numpy(), d_rad=d_rad.cpu().numpy())
    rp, pm = check_csr(w, res)
    check_forward(w, res, rp, pm)
    check_backward(w, res)


@pytest.mark.parametrize("name", ["n4096", "zipf"])
def test_backward_variants_agree(name):
    # the edge-order and CSR-order backward sum in different orders: both
    # within the tolerance of each other, each bitwise reproducible
    w = workloads.make_workload(name)
    dst, coup, rad, g = dev(w.dst), dev(w.coup), dev(w.rad), dev(w.grad_out)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    a = zs.zs_backward(g, coup, rad, dst, w.N)
    b = zs.zs_backward_csr(g, coup, rad, row_ptr, perm, w.N)
    b2 = zs.zs_backward_csr(g, coup, rad, row_ptr, perm, w.N)
    assert torch.equal(b[0], b2[0]) and torch.equal(b[1], b2[1])
    _, _, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    assert_close(a[0].cpu().numpy(), b[0].cpu().numpy(), adc, "d_coup edge vs csr", tol=2 * TOL)
    assert_close(a[1].cpu().numpy(), b[1].cpu().numpy(), adr, "d_rad edge vs csr", tol=2 * TOL)
    zs.zs_check_timeouts()
