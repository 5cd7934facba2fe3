"""Checks that pin an implementation of the zonal scatter to facts outside it.

Each check takes implementations as callables, so the same checks run on the
C oracle, on the torch composition and on deliberately broken copies (the
planted-mistake tests), and every plausible mistake must fail one of them.

    fwd(coup, rad, dst, N)        -> out (N, 16, C)
    bwd(g, coup, rad, dst, N)     -> (d_coup (E, 15), d_rad (E, 3, C))
    csr(dst, N)                   -> (row_ptr (N+1,), perm (E,), bad count)

Sources for the facts: deepmd-kit pull request "fused Triton zonal scatter for
the GIE head" -- section "What" (forward walks the stable destination CSR,
zero scalar row; backward gives the (E, 15) coupling and (E, 3, C) radial
gradients) and section "Boundary and layout contract" (row groups 3/5/7).
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


class PinFailure(AssertionError):
    pass


def _require(cond, msg):
    if not cond:
        raise PinFailure(msg)


# ---------------------------------------------------------------- fixtures


def hand_example():
    """Inputs and hand-computed values of tests/golden/hand_example.json."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        h = json.load(f)
    N, C = h["N"], h["C"]
    dst = np.array(h["dst"], np.int32)
    a = np.array(h["a"], np.float64)
    b = np.array(h["b"], np.float64)
    E = dst.shape[0]
    r = np.arange(15)
    s = np.array([0] * 3 + [1] * 5 + [2] * 7)
    c = np.arange(C)
    coup = ((r[None, :] + 1) * a[:, None]).astype(np.float32)
    rad = (b[:, None, None] * (10 * np.arange(3)[None, :, None] + c[None, None, :] + 1)).astype(np.float32)
    g = np.zeros((N, 16, C), np.float32)
    g[:, 0, :] = h["g_scalar_row"]
    g[:, 1:, :] = ((np.arange(N)[:, None, None] + 1) * (c[None, None, :] + 1)).astype(np.float32)
    del s, E
    return h, dst, coup, rad, g


def tiny_graph(seed, N, E, C, *, quantised=False, self_loops=True):
    """Small random graph.  quantised=True puts every value on a grid whose
    perturbation by +-2^-10 stays exact in fp32 (for finite differences)."""
    rng = np.random.default_rng(seed)
    dst = rng.integers(0, N, size=E).astype(np.int32)
    if not self_loops:
        pass
    if quantised:
        coup = (rng.integers(-2 ** 19, 2 ** 19, size=(E, 15)) / 2.0 ** 19).astype(np.float32)
        rad = (rng.integers(-2 ** 18, 2 ** 18, size=(E, 3, C)) / 2.0 ** 16).astype(np.float32)
    else:
        coup = rng.uniform(-1, 1, size=(E, 15)).astype(np.float32)
        rad = rng.standard_normal((E, 3, C)).astype(np.float32)
    g = rng.standard_normal((N, 16, C)).astype(np.float32)
    return dst, coup, rad, g


# ---------------------------------------------------------------- pins


def pin_golden(fwd, bwd, csr):
    h, dst, coup, rad, g = hand_example()
    N = h["N"]
    row_ptr, perm, bad = csr(dst, N)
    _require(list(np.asarray(row_ptr)) == h["row_ptr"], "golden row_ptr")
    _require(list(np.asarray(perm)) == h["perm"], "golden perm")
    _require(bad == 0, "golden bad count")
    out = np.asarray(fwd(coup, rad, dst, N))
    for (n, k, c), v, _ in h["out"]:
        _require(abs(out[n, k, c] - v) <= 1e-9 * max(1.0, abs(v)), f"golden out[{n},{k},{c}]={out[n, k, c]} != {v}")
    _require(np.all(out[:, 0, :] == 0), "golden scalar row")
    _require(np.all(out[1] == 0), "golden empty node")
    d_coup, d_rad = bwd(g, coup, rad, dst, N)
    d_coup = np.asarray(d_coup)
    d_rad = np.asarray(d_rad)
    for (e, r), v, _ in h["d_coup"]:
        _require(abs(d_coup[e, r] - v) <= 1e-9 * max(1.0, abs(v)), f"golden d_coup[{e},{r}]={d_coup[e, r]} != {v}")
    for (e, s, c), v, _ in h["d_rad"]:
        _require(abs(d_rad[e, s, c] - v) <= 1e-9 * max(1.0, abs(v)), f"golden d_rad[{e},{s},{c}]={d_rad[e, s, c]} != {v}")


def pin_csr_textbook(csr, seeds=(0, 1, 2, 3)):
    """CSR against numpy's stable argsort and bincount, and torch's stable sort."""
    import torch
    for seed in seeds:
        rng = np.random.default_rng(100 + seed)
        N = int(rng.integers(1, 300))
        E = int(rng.integers(0, 5000))
        dst = rng.integers(0, N, size=E).astype(np.int32)
        row_ptr, perm, bad = csr(dst, N)
        want_perm = np.argsort(dst, kind="stable").astype(np.int32)
        want_rp = np.concatenate([[0], np.cumsum(np.bincount(dst, minlength=N))]).astype(np.int32)
        t_perm = torch.sort(torch.from_numpy(dst.astype(np.int64)), stable=True).indices.numpy().astype(np.int32)
        _require(np.array_equal(want_perm, t_perm), "numpy and torch stable sorts disagree")
        _require(np.array_equal(np.asarray(perm), want_perm), f"perm != stable argsort (seed {seed})")
        _require(np.array_equal(np.asarray(row_ptr), want_rp), f"row_ptr != scan of bincount (seed {seed})")
        _require(bad == 0, "bad count on valid input")


def pin_csr_bad_dst(csr):
    """Out-of-range destinations: excluded from segments, appended in edge order."""
    dst = np.array([3, -1, 0, 7, 3, 0, 4, -5, 1], np.int32)   # N = 4 -> 4, 7, -1, -5 invalid
    N = 4
    row_ptr, perm, bad = csr(dst, N)
    valid = (dst >= 0) & (dst < N)
    keys = np.where(valid, dst, N)
    want_perm = np.argsort(keys, kind="stable").astype(np.int32)
    _require(bad == int((~valid).sum()), "bad count")
    _require(np.array_equal(np.asarray(perm), want_perm), "perm with bad destinations")
    want_rp = np.concatenate([[0], np.cumsum(np.bincount(dst[valid], minlength=N))])
    _require(np.array_equal(np.asarray(row_ptr), want_rp), "row_ptr with bad destinations")


def brute_forward(coup, rad, dst, N):
    """Pure-Python loops over every (node, edge) pair; no CSR, no index_add."""
    E, C = rad.shape[0], rad.shape[2]
    out = np.zeros((N, 16, C))
    for n in range(N):
        for e in range(E):
            if dst[e] != n:
                continue
            for r in range(15):
                s = 0 if r <= 2 else (1 if r <= 7 else 2)
                for c in range(C):
                    out[n, 1 + r, c] += float(coup[e, r]) * float(rad[e, s, c])
    return out


def brute_backward(g, coup, rad, dst, N):
    E, C = rad.shape[0], rad.shape[2]
    d_coup = np.zeros((E, 15))
    d_rad = np.zeros((E, 3, C))
    for e in range(E):
        n = int(dst[e])
        if n < 0 or n >= N:
            continue
        for r in range(15):
            s = 0 if r <= 2 else (1 if r <= 7 else 2)
            for c in range(C):
                d_coup[e, r] += float(g[n, 1 + r, c]) * float(rad[e, s, c])
                d_rad[e, s, c] += float(g[n, 1 + r, c]) * float(coup[e, r])
    return d_coup, d_rad


def pin_brute_force(fwd, bwd, cases=((5, 17, 3, 0), (8, 32, 4, 1), (1, 6, 2, 2), (6, 0, 3, 3))):
    for N, E, C, seed in cases:
        dst, coup, rad, g = tiny_graph(seed, N, E, C)
        out = np.asarray(fwd(coup, rad, dst, N))
        ref = brute_forward(coup, rad, dst, N)
        _require(out.shape == ref.shape and np.allclose(out, ref, rtol=1e-12, atol=1e-12), f"forward vs brute force {N, E, C}")
        dc, dr = bwd(g, coup, rad, dst, N)
        rdc, rdr = brute_backward(g, coup, rad, dst, N)
        _require(np.allclose(dc, rdc, rtol=1e-12, atol=1e-12), f"d_coup vs brute force {N, E, C}")
        _require(np.allclose(dr, rdr, rtol=1e-12, atol=1e-12), f"d_rad vs brute force {N, E, C}")


def pin_closed_forms(fwd, bwd):
    rng = np.random.default_rng(7)
    # one edge e -> n: out[n,1+r,c] = coup*rad exactly
    N, C = 4, 5
    coup = rng.uniform(-1, 1, (1, 15)).astype(np.float32)
    rad = rng.standard_normal((1, 3, C)).astype(np.float32)
    dst = np.array([2], np.int32)
    out = np.asarray(fwd(coup, rad, dst, N))
    for r in range(15):
        s = 0 if r < 3 else (1 if r < 8 else 2)
        _require(np.array_equal(out[2, 1 + r], coup[0, r].astype(np.float64) * rad[0, s].astype(np.float64)),
                 f"single edge row {r}")
    _require(np.all(out[[0, 1, 3]] == 0), "single edge other nodes")
    # all-ones operands: out = in-degree, d_coup = sum_c g, d_rad = sum over the slot's rows of g
    N, E, C = 9, 200, 6
    dst = rng.integers(0, N, E).astype(np.int32)
    ones_c = np.ones((E, 15), np.float32)
    ones_r = np.ones((E, 3, C), np.float32)
    out = np.asarray(fwd(ones_c, ones_r, dst, N))
    indeg = np.bincount(dst, minlength=N).astype(np.float64)
    _require(np.array_equal(out[:, 1:, :], np.broadcast_to(indeg[:, None, None], (N, 15, C))), "ones -> in-degree")
    _require(np.all(out[:, 0, :] == 0), "ones scalar row")
    g = rng.standard_normal((N, 16, C)).astype(np.float32)
    dc, dr = bwd(g, ones_c, ones_r, dst, N)
    gd = g[dst].astype(np.float64)
    _require(np.allclose(dc, gd[:, 1:, :].sum(2), rtol=1e-13, atol=1e-13), "ones -> d_coup = sum_c g")
    want = np.stack([gd[:, 1:4].sum(1), gd[:, 4:9].sum(1), gd[:, 9:16].sum(1)], axis=1)
    _require(np.allclose(dr, want, rtol=1e-13, atol=1e-13), "ones -> d_rad = sum of the slot's g rows")
    # no edges: all zeros
    out = np.asarray(fwd(np.zeros((0, 15), np.float32), np.zeros((0, 3, C), np.float32), np.zeros(0, np.int32), N))
    _require(out.shape == (N, 16, C) and np.all(out == 0), "E = 0")


def pin_finite_differences(fwd, bwd, cases=((4, 12, 3, 11), (7, 25, 2, 12))):
    """Central differences of L = <g, fwd> with perturbations exact in fp32."""
    h = 2.0 ** -10
    for N, E, C, seed in cases:
        dst, coup, rad, g = tiny_graph(seed, N, E, C, quantised=True)
        g64 = g.astype(np.float64)

        def L(cp, rd):
            return float(np.sum(g64 * np.asarray(fwd(cp, rd, dst, N))))

        dc, dr = bwd(g, coup, rad, dst, N)
        dc = np.asarray(dc)
        dr = np.asarray(dr)
        scale = 1.0 + np.abs(dc).max()
        for e in range(E):
            for r in (0, 2, 3, 7, 8, 14):
                p = coup.copy(); p[e, r] += np.float32(h)
                m = coup.copy(); m[e, r] -= np.float32(h)
                _require(float(p[e, r]) - float(m[e, r]) == 2 * h, "perturbation not exact")
                fd = (L(p, rad) - L(m, rad)) / (2 * h)
                _require(abs(fd - dc[e, r]) <= 1e-9 * scale, f"FD d_coup[{e},{r}] {fd} vs {dc[e, r]}")
        scale = 1.0 + np.abs(dr).max()
        for e in range(0, E, 3):
            for s in range(3):
                for c in range(C):
                    p = rad.copy(); p[e, s, c] += np.float32(h)
                    m = rad.copy(); m[e, s, c] -= np.float32(h)
                    fd = (L(coup, p) - L(coup, m)) / (2 * h)
                    _require(abs(fd - dr[e, s, c]) <= 1e-9 * scale, f"FD d_rad[{e},{s},{c}] {fd} vs {dr[e, s, c]}")


def pin_adjoint(fwd, bwd, cases=((13, 300, 5, 21), (50, 2000, 8, 22))):
    """<g, fwd(coup, rad)> = <d_coup, coup> = <d_rad, rad> (the op is bilinear)."""
    for N, E, C, seed in cases:
        dst, coup, rad, g = tiny_graph(seed, N, E, C)
        out = np.asarray(fwd(coup, rad, dst, N))
        dc, dr = bwd(g, coup, rad, dst, N)
        a = float(np.sum(g.astype(np.float64)[:, 1:] * out[:, 1:]))
        b = float(np.sum(np.asarray(dc) * coup.astype(np.float64)))
        c = float(np.sum(np.asarray(dr) * rad.astype(np.float64)))
        scale = float(np.sum(np.abs(g.astype(np.float64)[dst][:, 1:] * coup.astype(np.float64)[:, :, None]
                                    * rad.astype(np.float64)[:, [0] * 3 + [1] * 5 + [2] * 7, :])))
        _require(abs(a - b) <= 1e-12 * scale and abs(a - c) <= 1e-12 * scale, f"adjoint {a} {b} {c}")
        # the scalar row of g must not matter
        g2 = g.copy(); g2[:, 0, :] = 1e6
        dc2, dr2 = bwd(g2, coup, rad, dst, N)
        _require(np.array_equal(dc2, dc) and np.array_equal(dr2, dr), "g scalar row is read")


def pin_conservation(fwd, cases=((30, 900, 4, 31),)):
    """Sum over nodes of out equals the sum over edges of coup*rad (no scatter)."""
    for N, E, C, seed in cases:
        dst, coup, rad, _ = tiny_graph(seed, N, E, C)
        out = np.asarray(fwd(coup, rad, dst, N))
        tot = out[:, 1:, :].sum(0)
        c64 = coup.astype(np.float64)
        r64 = rad.astype(np.float64)
        want = np.concatenate([
            np.einsum("er,ec->rc", c64[:, 0:3], r64[:, 0]),
            np.einsum("er,ec->rc", c64[:, 3:8], r64[:, 1]),
            np.einsum("er,ec->rc", c64[:, 8:15], r64[:, 2]),
        ])
        _require(np.allclose(tot, want, rtol=1e-12, atol=1e-10), "conservation")
        _require(np.all(out[:, 0, :] == 0), "scalar row")
        empty = np.setdiff1d(np.arange(N), dst)
        _require(np.all(out[empty] == 0), "zero in-degree rows")


ALL_PINS = ("golden", "csr_textbook", "csr_bad_dst", "brute_force", "closed_forms",
            "finite_differences", "adjoint", "conservation")


def run_all(fwd, bwd, csr):
    """Run every pin; return the names of those that failed."""
    failed = []
    for name, fn in (
        ("golden", lambda: pin_golden(fwd, bwd, csr)),
        ("csr_textbook", lambda: pin_csr_textbook(csr)),
        ("csr_bad_dst", lambda: pin_csr_bad_dst(csr)),
        ("brute_force", lambda: pin_brute_force(fwd, bwd)),
        ("closed_forms", lambda: pin_closed_forms(fwd, bwd)),
        ("finite_differences", lambda: pin_finite_differences(fwd, bwd)),
        ("adjoint", lambda: pin_adjoint(fwd, bwd)),
        ("conservation", lambda: pin_conservation(fwd)),
    ):
        try:
            fn()
        except PinFailure:
            failed.append(name)
    return failed


# ---------------------------------------------------------------- general lmax
#
# The ladder of degree lmax: D = (lmax+1)^2 node rows, the scalar row then
# degree groups of 2l+1 zonal rows (l = 1..lmax), radial slot l - 1 (the lmax
# = 3 case is the pages' 3/5/7).  The slot list is built here by counting
# rows degree by degree, independently of any implementation's formula.


def ladder_slots(lmax):
    slots = []
    for l in range(1, lmax + 1):
        slots += [l - 1] * (2 * l + 1)
    return np.array(slots, np.int64)


def tiny_graph_l(seed, N, E, C, lmax, *, quantised=False):
    rng = np.random.default_rng(1000 * lmax + seed)
    R = (lmax + 1) ** 2 - 1
    dst = rng.integers(0, N, size=E).astype(np.int32)
    if quantised:
        coup = (rng.integers(-2 ** 19, 2 ** 19, size=(E, R)) / 2.0 ** 19).astype(np.float32)
        rad = (rng.integers(-2 ** 18, 2 ** 18, size=(E, lmax, C)) / 2.0 ** 16).astype(np.float32)
    else:
        coup = rng.uniform(-1, 1, size=(E, R)).astype(np.float32)
        rad = rng.standard_normal((E, lmax, C)).astype(np.float32)
    g = rng.standard_normal((N, R + 1, C)).astype(np.float32)
    return dst, coup, rad, g


def brute_forward_l(coup, rad, dst, N, lmax):
    E, C = rad.shape[0], rad.shape[2]
    slots = ladder_slots(lmax)
    out = np.zeros((N, len(slots) + 1, C))
    for n in range(N):
        for e in range(E):
            if dst[e] != n:
                continue
            for r, s in enumerate(slots):
                for c in range(C):
                    out[n, 1 + r, c] += float(coup[e, r]) * float(rad[e, s, c])
    return out


def brute_backward_l(g, coup, rad, dst, N, lmax):
    E, C = rad.shape[0], rad.shape[2]
    slots = ladder_slots(lmax)
    d_coup = np.zeros((E, len(slots)))
    d_rad = np.zeros((E, lmax, C))
    for e in range(E):
        n = int(dst[e])
        if n < 0 or n >= N:
            continue
        for r, s in enumerate(slots):
            for c in range(C):
                d_coup[e, r] += float(g[n, 1 + r, c]) * float(rad[e, s, c])
                d_rad[e, s, c] += float(g[n, 1 + r, c]) * float(coup[e, r])
    return d_coup, d_rad


def pin_general_lmax(fwd, bwd, lmax):
    """Brute force, closed forms, adjoint identity and finite differences at lmax."""
    R = (lmax + 1) ** 2 - 1
    slots = ladder_slots(lmax)
    _require(len(slots) == R, "ladder size")
    # brute force over every (node, edge) pair
    for N, E, C, seed in ((5, 14, 3, 0), (3, 9, 2, 1)):
        dst, coup, rad, g = tiny_graph_l(seed, N, E, C, lmax)
        out = np.asarray(fwd(coup, rad, dst, N))
        _require(out.shape == (N, R + 1, C), f"lmax {lmax} output shape {out.shape}")
        _require(np.allclose(out, brute_forward_l(coup, rad, dst, N, lmax), rtol=1e-12, atol=1e-12),
                 f"lmax {lmax} forward vs brute force")
        dc, dr = bwd(g, coup, rad, dst, N)
        rdc, rdr = brute_backward_l(g, coup, rad, dst, N, lmax)
        _require(np.shape(dc) == rdc.shape and np.shape(dr) == rdr.shape, f"lmax {lmax} gradient shapes")
        _require(np.allclose(dc, rdc, rtol=1e-12, atol=1e-12), f"lmax {lmax} d_coup vs brute force")
        _require(np.allclose(dr, rdr, rtol=1e-12, atol=1e-12), f"lmax {lmax} d_rad vs brute force")
    # all-ones operands: out = in-degree; d_coup = sum_c g; d_rad = the slot's rows of g summed
    rng = np.random.default_rng(70 + lmax)
    N, E, C = 7, 150, 4
    dst = rng.integers(0, N, E).astype(np.int32)
    out = np.asarray(fwd(np.ones((E, R), np.float32), np.ones((E, lmax, C), np.float32), dst, N))
    indeg = np.bincount(dst, minlength=N).astype(np.float64)
    _require(np.array_equal(out[:, 1:, :], np.broadcast_to(indeg[:, None, None], (N, R, C))), f"lmax {lmax} ones")
    _require(np.all(out[:, 0, :] == 0), f"lmax {lmax} scalar row")
    g = rng.standard_normal((N, R + 1, C)).astype(np.float32)
    dc, dr = bwd(g, np.ones((E, R), np.float32), np.ones((E, lmax, C), np.float32), dst, N)
    gd = g[dst].astype(np.float64)
    _require(np.allclose(dc, gd[:, 1:, :].sum(2), rtol=1e-13, atol=1e-13), f"lmax {lmax} ones d_coup")
    first = 0
    for l in range(1, lmax + 1):
        rows = slice(1 + first, 1 + first + 2 * l + 1)
        _require(np.allclose(np.asarray(dr)[:, l - 1], gd[:, rows].sum(1), rtol=1e-13, atol=1e-13),
                 f"lmax {lmax} ones d_rad degree {l}")
        first += 2 * l + 1
    # adjoint identity (the op is bilinear)
    dst, coup, rad, g = tiny_graph_l(5, 11, 200, 3, lmax)
    out = np.asarray(fwd(coup, rad, dst, 11))
    dc, dr = bwd(g, coup, rad, dst, 11)
    a = float(np.sum(g.astype(np.float64)[:, 1:] * out[:, 1:]))
    b = float(np.sum(np.asarray(dc) * coup.astype(np.float64)))
    c = float(np.sum(np.asarray(dr) * rad.astype(np.float64)))
    scale = float(np.sum(np.abs(g.astype(np.float64)[dst][:, 1:] * coup.astype(np.float64)[:, :, None]
                                * rad.astype(np.float64)[:, slots, :])))
    _require(abs(a - b) <= 1e-12 * scale and abs(a - c) <= 1e-12 * scale, f"lmax {lmax} adjoint {a} {b} {c}")
    # central differences with perturbations exact in fp32
    h = 2.0 ** -10
    N, E, C = 3, 6, 2
    dst, coup, rad, g = tiny_graph_l(9, N, E, C, lmax, quantised=True)
    g64 = g.astype(np.float64)

    def L(cp, rd):
        return float(np.sum(g64 * np.asarray(fwd(cp, rd, dst, N))))

    dc, dr = bwd(g, coup, rad, dst, N)
    dc = np.asarray(dc)
    dr = np.asarray(dr)
    scale = 1.0 + max(np.abs(dc).max(), np.abs(dr).max())
    for e in range(E):
        for r in sorted({0, R // 2, R - 1}):
            p = coup.copy(); p[e, r] += np.float32(h)
            m = coup.copy(); m[e, r] -= np.float32(h)
            fd = (L(p, rad) - L(m, rad)) / (2 * h)
            _require(abs(fd - dc[e, r]) <= 1e-9 * scale, f"lmax {lmax} FD d_coup[{e},{r}]")
        for s in range(lmax):
            p = rad.copy(); p[e, s, 0] += np.float32(h)
            m = rad.copy(); m[e, s, 0] -= np.float32(h)
            fd = (L(coup, p) - L(coup, m)) / (2 * h)
            _require(abs(fd - dr[e, s, 0]) <= 1e-9 * scale, f"lmax {lmax} FD d_rad[{e},{s},0]")


# ---------------------------------------------------------------- node factor
#
# The degree normalisation the pages apply to the operator's output (section
# "What", third bullet): out[n] = s[n] * (operator output)[n], s one factor
# per node; reading: a node without edges stays zero whatever s[n].
#   fwd_s(coup, rad, dst, N, s)            -> (out, out_raw)
#   bwd_s(g, coup, rad, dst, N, s, raw)    -> (d_coup, d_rad, d_scale)


def pin_node_factor(fwd_s, bwd_s):
    rng = np.random.default_rng(404)
    # s = 1 is the plain operator, by brute force
    N, E, C = 6, 20, 3
    dst, coup, rad, g = tiny_graph(41, N, E, C)
    out, raw = fwd_s(coup, rad, dst, N, np.ones(N, np.float32))
    ref = brute_forward(coup, rad, dst, N)
    _require(np.allclose(out, ref, rtol=1e-12, atol=1e-12) and np.allclose(raw, ref, rtol=1e-12, atol=1e-12),
             "node factor 1 vs brute force")
    # each node's rows scale by its factor; a node without edges is zero even for s = inf
    dst = (dst % (N - 1)).astype(np.int32)          # node N-1 gets no edge
    ref = brute_forward(coup, rad, dst, N)
    s = rng.uniform(-2, 2, N).astype(np.float32)
    empty = np.setdiff1d(np.arange(N), dst)
    s[empty[0]] = np.inf
    out, raw = fwd_s(coup, rad, dst, N, s)
    has = np.isin(np.arange(N), dst)
    want = np.zeros_like(ref)
    want[has] = s.astype(np.float64)[has, None, None] * ref[has]
    _require(np.allclose(out, want, rtol=1e-12, atol=1e-12), "node factor scaling")
    _require(np.all(np.asarray(out)[empty] == 0), "node without edges under its factor")
    # trilinear adjoint: <g, out> = <d_coup, coup> = <d_rad, rad> = <d_scale, s>
    N, E, C = 17, 400, 4
    dst, coup, rad, g = tiny_graph(42, N, E, C)
    s = rng.uniform(0.1, 2, N).astype(np.float32)
    out, raw = fwd_s(coup, rad, dst, N, s)
    dc, dr, ds = bwd_s(g, coup, rad, dst, N, s, raw)
    a = float(np.sum(g.astype(np.float64)[:, 1:] * np.asarray(out)[:, 1:]))
    b = float(np.sum(np.asarray(dc) * coup.astype(np.float64)))
    c = float(np.sum(np.asarray(dr) * rad.astype(np.float64)))
    d = float(np.sum(np.asarray(ds) * s.astype(np.float64)))
    scale = float(np.sum(np.abs(g.astype(np.float64)[:, 1:] * np.asarray(out)[:, 1:]))) + 1.0
    _require(max(abs(a - b), abs(a - c), abs(a - d)) <= 1e-11 * scale, f"node factor adjoint {a} {b} {c} {d}")
    # central differences in s (the output is linear in s)
    h = 2.0 ** -8
    N, E, C = 5, 30, 2
    dst, coup, rad, g = tiny_graph(43, N, E, C, quantised=True)
    s = (rng.integers(1, 64, N) / 16.0).astype(np.float32)
    out, raw = fwd_s(coup, rad, dst, N, s)
    _, _, ds = bwd_s(g, coup, rad, dst, N, s, raw)
    g64 = g.astype(np.float64)
    for n in range(N):
        p = s.copy(); p[n] += np.float32(h)
        m = s.copy(); m[n] -= np.float32(h)
        fd = (float(np.sum(g64 * np.asarray(fwd_s(coup, rad, dst, N, p)[0]))) -
              float(np.sum(g64 * np.asarray(fwd_s(coup, rad, dst, N, m)[0])))) / (2 * h)
        _require(abs(fd - float(np.asarray(ds)[n])) <= 1e-9 * (1.0 + abs(fd)), f"FD d_scale[{n}]")
