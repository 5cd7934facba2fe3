"""The CPU oracle against facts outside itself, and planted mistakes caught.

Runs without a GPU.  See tests/pins.py for what each pin checks.
"""
import numpy as np
import pytest

import oracle
from oracle import composition
from equivariant_interatomic_potential_gb300 import workloads
import pins


# ----------------------------------------------------------- adapters

def a_fwd(coup, rad, dst, N):
    row_ptr, perm, _ = oracle.build_csr(dst, N)
    out, _ = oracle.forward(coup, rad, row_ptr, perm, N)
    return out


def a_bwd(g, coup, rad, dst, N):
    dc, dr, _, _ = oracle.backward(g, coup, rad, dst, N)
    return dc, dr


def a_csr(dst, N):
    return oracle.build_csr(dst, N)


def b_fwd(coup, rad, dst, N):
    return composition.forward(coup, rad, dst, N)


def b_bwd(g, coup, rad, dst, N):
    return composition.backward(g, coup, rad, dst, N)


# ----------------------------------------------------------- pins on both variants

@pytest.mark.parametrize("pin", pins.ALL_PINS)
def test_oracle_a_pins(pin):
    fn = {
        "golden": lambda: pins.pin_golden(a_fwd, a_bwd, a_csr),
        "csr_textbook": lambda: pins.pin_csr_textbook(a_csr),
        "csr_bad_dst": lambda: pins.pin_csr_bad_dst(a_csr),
        "brute_force": lambda: pins.pin_brute_force(a_fwd, a_bwd),
        "closed_forms": lambda: pins.pin_closed_forms(a_fwd, a_bwd),
        "finite_differences": lambda: pins.pin_finite_differences(a_fwd, a_bwd),
        "adjoint": lambda: pins.pin_adjoint(a_fwd, a_bwd),
        "conservation": lambda: pins.pin_conservation(a_fwd),
    }[pin]
    fn()


def test_oracle_b_pins():
    assert pins.run_all(b_fwd, b_bwd, a_csr) == []


def test_slot_map_matches_row_groups():
    # rows 0-2 -> degree 1, 3-7 -> degree 2, 8-14 -> degree 3 (row groups 3/5/7)
    assert [oracle.slot_of_row(r) for r in range(15)] == [0] * 3 + [1] * 5 + [2] * 7
    assert composition.slot_index().tolist() == [0] * 3 + [1] * 5 + [2] * 7
    assert composition.row_groups(3) == composition.ROW_GROUPS
    # further degrees continue the ladder: 9 rows of degree 4, 11 of degree 5
    assert [oracle.slot_of_row(r) for r in range(35)] == pins.ladder_slots(5).tolist()


@pytest.mark.parametrize("lmax", [1, 2, 3, 4, 5])
def test_general_lmax_pins(lmax):
    pins.pin_general_lmax(a_fwd, a_bwd, lmax)
    pins.pin_general_lmax(b_fwd, b_bwd, lmax)


def test_general_lmax_a_matches_composition():
    for lmax in (1, 2, 4, 5):
        w = workloads.make_random(40, 3000, 6, seed=lmax, lmax=lmax)
        out_a = a_fwd(w.coup, w.rad, w.dst, w.N)
        out_b = b_fwd(w.coup, w.rad, w.dst, w.N)
        _, absum = oracle.forward(w.coup, w.rad, *oracle.build_csr(w.dst, w.N)[:2], w.N)
        err, bad = oracle.normalised_error(out_a, out_b, absum)
        assert err <= 1e-12 and bad == 0
        dca, dra = a_bwd(w.grad_out, w.coup, w.rad, w.dst, w.N)
        dcb, drb = b_bwd(w.grad_out, w.coup, w.rad, w.dst, w.N)
        assert np.allclose(dca, dcb, rtol=1e-12, atol=1e-12) and np.allclose(dra, drb, rtol=1e-12, atol=1e-12)


def _general_groups_mutant(groups):
    # the composition with the degree-4/5 groups resized (rows move to the wrong slot)
    def fwd(cp, rd, d, N):
        old = composition.row_groups
        composition.row_groups = lambda lmax=3: groups[:lmax]
        try:
            return composition.forward(cp, rd, d, N)
        finally:
            composition.row_groups = old

    def bwd(g, cp, rd, d, N):
        old = composition.row_groups
        composition.row_groups = lambda lmax=3: groups[:lmax]
        try:
            return composition.backward(g, cp, rd, d, N)
        finally:
            composition.row_groups = old
    return fwd, bwd


@pytest.mark.parametrize("groups", [(3, 5, 7, 10, 10), (3, 5, 8, 8, 11), (3, 5, 7, 11, 9)])
def test_general_lmax_planted_groups_caught(groups):
    fwd, bwd = _general_groups_mutant(groups)
    with pytest.raises(pins.PinFailure):
        pins.pin_general_lmax(fwd, bwd, 5)


# ----------------------------------------------------------- A against B

@pytest.mark.parametrize("case", ["tiny", "n1000", "odd40", "selfloops_C3", "hot_node"])
def test_variant_a_matches_composition(case):
    if case in ("tiny", "n1000"):
        w = workloads.make_workload(case)
    elif case == "odd40":
        w = workloads.make_random(33, 777, 40, seed=5)
    elif case == "selfloops_C3":
        w = workloads.make_random(17, 900, 3, seed=6, self_loops=True)
    else:
        w = workloads.make_random(50, 3000, 8, seed=7, hot_node=3, hot_fraction=0.6)
    row_ptr, perm, bad = oracle.build_csr(w.dst, w.N)
    assert bad == 0
    out, absum = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N)
    ref = composition.forward(w.coup, w.rad, w.dst, w.N)
    err, bz = oracle.normalised_error(out, ref, absum)
    assert err <= 1e-12 and bz == 0
    assert np.all(out[:, 0, :] == 0)
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    rdc, rdr = composition.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    e1, z1 = oracle.normalised_error(dc, rdc, adc)
    e2, z2 = oracle.normalised_error(dr, rdr, adr)
    assert e1 <= 1e-12 and e2 <= 1e-12 and z1 == 0 and z2 == 0


def test_sampled_entry_points_match_full():
    w = workloads.make_workload("tiny")
    row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
    out, absum = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N)
    nodes = np.array([5, 0, 63, 5], np.int32)
    o2, a2 = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N, nodes=nodes)
    assert np.array_equal(o2, out[nodes]) and np.array_equal(a2, absum[nodes])
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    edges = np.array([0, 2047, 17, 17], np.int64)
    dc2, dr2, adc2, adr2 = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N, edges=edges)
    assert np.array_equal(dc2, dc[edges]) and np.array_equal(dr2, dr[edges])
    assert np.array_equal(adc2, adc[edges]) and np.array_equal(adr2, adr[edges])


def test_zipf_zero_in_degree_rows_are_zero():
    w = workloads.make_workload("zipf")
    row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
    deg = np.diff(row_ptr)
    assert (deg == 0).sum() == 205
    nodes = np.nonzero(deg == 0)[0].astype(np.int32)
    out, absum = oracle.forward(w.coup, w.rad, row_ptr, perm, w.N, nodes=nodes)
    assert np.all(out == 0) and np.all(absum == 0)


def test_normalised_error_rules():
    ref = np.array([1.0, 0.0, 2.0])
    absum = np.array([1.0, 0.0, 4.0])
    assert oracle.normalised_error(np.array([1.0, 0.0, 2.0]), ref, absum) == (0.0, 0)
    assert oracle.normalised_error(np.array([1.0, 1e-30, 2.0]), ref, absum)[1] == 1
    assert oracle.normalised_error(np.array([np.nan, 0.0, 2.0]), ref, absum)[0] == np.inf
    assert oracle.normalised_error(np.array([1.0, 0.0, 2.4]), ref, absum)[0] == pytest.approx(0.1)


# ----------------------------------------------------------- planted mistakes

def _mut_slot_reversed():
    return (lambda cp, rd, d, N: a_fwd(cp, np.ascontiguousarray(rd[:, ::-1, :]), d, N),
            lambda g, cp, rd, d, N: tuple(x if i == 0 else x[:, ::-1, :] for i, x in
                                          enumerate(a_bwd(g, cp, np.ascontiguousarray(rd[:, ::-1, :]), d, N))),
            a_csr)


def _mut_groups(groups):
    # the composition with its row grouping replaced
    def patched(call):
        old = composition.row_groups
        composition.row_groups = lambda lmax=3: groups
        try:
            return call()
        finally:
            composition.row_groups = old

    def fwd(cp, rd, d, N):
        return patched(lambda: composition.forward(cp, rd, d, N))

    def bwd(g, cp, rd, d, N):
        return patched(lambda: composition.backward(g, cp, rd, d, N))
    return fwd, bwd, a_csr


def _mut_drop_last_edge():
    def fwd(cp, rd, d, N):
        row_ptr, perm, _ = oracle.build_csr(d, N)
        d2 = np.array(d, np.int32, copy=True)
        for n in range(N):
            if row_ptr[n + 1] > row_ptr[n]:
                d2[perm[row_ptr[n + 1] - 1]] = -1
        return a_fwd(cp, rd, d2, N)
    return fwd, a_bwd, a_csr


def _mut_sign_drad():
    return a_fwd, (lambda g, cp, rd, d, N: (a_bwd(g, cp, rd, d, N)[0], -a_bwd(g, cp, rd, d, N)[1])), a_csr


def _mut_g_row_shift():
    def bwd(g, cp, rd, d, N):
        g2 = np.array(g, copy=True)
        g2[:, 1:, :] = g[:, :-1, :]
        return a_bwd(g2, cp, rd, d, N)
    return a_fwd, bwd, a_csr


def _mut_scalar_row():
    def fwd(cp, rd, d, N):
        out = a_fwd(cp, rd, d, N).copy()
        out[:, 0, :] = out[:, 1, :]
        return out
    return fwd, a_bwd, a_csr


def _mut_unstable_csr():
    def csr(d, N):
        row_ptr, perm, bad = oracle.build_csr(d, N)
        perm = perm.copy()
        for n in range(N):
            perm[row_ptr[n]:row_ptr[n + 1]] = perm[row_ptr[n]:row_ptr[n + 1]][::-1]
        return row_ptr, perm, bad
    return a_fwd, a_bwd, csr


def _mut_inclusive_scan():
    def csr(d, N):
        row_ptr, perm, bad = oracle.build_csr(d, N)
        rp = np.concatenate([row_ptr[1:], row_ptr[-1:]])
        return rp, perm, bad
    return a_fwd, a_bwd, csr


def _mut_clamped_bad_dst():
    def csr(d, N):
        d2 = np.clip(np.asarray(d), 0, max(N - 1, 0)).astype(np.int32)
        return oracle.build_csr(d2, N)
    return a_fwd, a_bwd, csr


def _mut_transposed_rad():
    def t(rd):
        E, S, C = rd.shape
        return np.ascontiguousarray(rd.reshape(E, C, S).transpose(0, 2, 1))
    return (lambda cp, rd, d, N: a_fwd(cp, t(rd), d, N),
            lambda g, cp, rd, d, N: a_bwd(g, cp, t(rd), d, N), a_csr)


def _mut_drad_uses_rad():
    # radial gradient formed with the radial operand in place of the coupling
    def bwd(g, cp, rd, d, N):
        dc, _ = a_bwd(g, cp, rd, d, N)
        E, _, C = rd.shape
        dr2 = np.zeros((E, 3, C))
        gd = np.asarray(g, np.float64)[np.asarray(d)]
        for s, rows in enumerate((range(0, 3), range(3, 8), range(8, 15))):
            for r in rows:
                dr2[:, s, :] += gd[:, 1 + r, :] * rd[:, s, :]
        return dc, dr2
    return a_fwd, bwd, a_csr


def _mut_fwd_uses_src_order_sum_twice():
    # the first edge of every node counted twice
    def fwd(cp, rd, d, N):
        out = a_fwd(cp, rd, d, N).copy()
        row_ptr, perm, _ = oracle.build_csr(d, N)
        for n in range(N):
            if row_ptr[n + 1] > row_ptr[n]:
                e = perm[row_ptr[n]]
                one = np.zeros(1, np.int32)
                o1, _ = oracle.forward(cp[e:e + 1], rd[e:e + 1], np.array([0, 1], np.int32), one, 1)
                out[n] += o1[0]
        return out
    return fwd, a_bwd, a_csr


MUTANTS = {
    "slot_order_reversed": _mut_slot_reversed,
    "row_groups_5_5_5": lambda: _mut_groups((5, 5, 5)),
    "row_groups_4_4_7": lambda: _mut_groups((4, 4, 7)),
    "row_groups_3_6_6": lambda: _mut_groups((3, 6, 6)),
    "dropped_last_edge": _mut_drop_last_edge,
    "d_rad_sign": _mut_sign_drad,
    "g_row_off_by_one": _mut_g_row_shift,
    "scalar_row_nonzero": _mut_scalar_row,
    "unstable_csr": _mut_unstable_csr,
    "inclusive_scan": _mut_inclusive_scan,
    "clamped_bad_dst": _mut_clamped_bad_dst,
    "transposed_rad": _mut_transposed_rad,
    "d_rad_uses_rad": _mut_drad_uses_rad,
    "first_edge_twice": _mut_fwd_uses_src_order_sum_twice,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    fwd, bwd, csr = MUTANTS[name]()
    failed = pins.run_all(fwd, bwd, csr)
    assert failed, f"planted mistake {name} passed every pin"


# ----------------------------------------------------------- node factor


def a_fwd_s(coup, rad, dst, N, s):
    row_ptr, perm, _ = oracle.build_csr(dst, N)
    out, _, raw, _ = oracle.forward_scaled(coup, rad, row_ptr, perm, N, s)
    return out, raw


def a_bwd_s(g, coup, rad, dst, N, s, raw):
    dc, dr, ds, _, _, _ = oracle.backward_scaled(g, coup, rad, dst, N, s, raw)
    return dc, dr, ds


def test_node_factor_pins():
    pins.pin_node_factor(a_fwd_s, a_bwd_s)


def test_node_factor_oracle_matches_autograd_composition():
    for lmax, C in ((3, 5), (2, 3)):
        w = workloads.make_random(30, 900, C, seed=55 + lmax, lmax=lmax)
        s = np.random.default_rng(lmax).uniform(-1.5, 1.5, w.N).astype(np.float32)
        row_ptr, perm, _ = oracle.build_csr(w.dst, w.N)
        out, _, raw, _ = oracle.forward_scaled(w.coup, w.rad, row_ptr, perm, w.N, s)
        dc, dr, ds, _, _, _ = oracle.backward_scaled(w.grad_out, w.coup, w.rad, w.dst, w.N, s, raw)
        out_b, dc_b, dr_b, ds_b = composition.scaled_with_autograd(w.coup, w.rad, w.dst, w.N, s, w.grad_out)
        for x, y in ((out, out_b), (dc, dc_b), (dr, dr_b), (ds, ds_b)):
            assert np.allclose(x, y, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("mistake", ["d_scale_from_scaled_out", "gradients_unscaled", "factor_on_empty_nodes"])
def test_node_factor_planted_mistakes_caught(mistake):
    def fwd(coup, rad, dst, N, s):
        out, raw = a_fwd_s(coup, rad, dst, N, s)
        if mistake == "factor_on_empty_nodes":
            out = np.asarray(s, np.float64)[:, None, None] * np.asarray(raw)
        return out, raw

    def bwd(g, coup, rad, dst, N, s, raw):
        dc, dr, ds = a_bwd_s(g, coup, rad, dst, N, s, raw)
        if mistake == "d_scale_from_scaled_out":
            ds = ds * np.asarray(s, np.float64)
        if mistake == "gradients_unscaled":
            dc, dr = a_bwd(g, coup, rad, dst, N)
        return dc, dr, ds
    with pytest.raises((pins.PinFailure, FloatingPointError)):
        with np.errstate(invalid="raise"):
            pins.pin_node_factor(fwd, bwd)


def test_oracle_threads_do_not_change_results():
    w = workloads.make_random(300, 20000, 8, seed=91, hot_node=4, hot_fraction=0.3)
    rp, pm, _ = oracle.build_csr(w.dst, w.N)
    one = oracle.forward(w.coup, w.rad, rp, pm, w.N), oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    oracle.set_threads(4)
    try:
        many = oracle.forward(w.coup, w.rad, rp, pm, w.N), oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    finally:
        oracle.set_threads(1)
    for a, b in zip(one[0] + one[1], many[0] + many[1]):
        assert np.array_equal(a, b)
