"""CPU oracle for the GIE zonal scatter.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA path, and the
product never calls it.

Two independent formulations of the same definitions (deepmd-kit pull request
"fused Triton zonal scatter for the GIE head", section "What"):

* variant A (``zs_oracle.c``, fp64, sequential): stable CSR by counting sort,
  forward as a per-node walk of that CSR in order, backward as direct loops;
  every value comes with the sum of |terms| that formed it.
* variant B (``composition.py``, torch CPU fp64): the reference composition the
  page replaces -- broadcast the coupling over each degree's radial rows into
  a materialised (E, 15, C) message, then ``index_add_`` it onto the
  destinations; its backward is the same composition's adjoint.

Pins against things other than the oracle itself live in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zs_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_zs.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no GPU code involved)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_build_csr.restype = ctypes.c_int64
            lib.oracle_build_csr.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P]
            lib.oracle_forward.restype = None
            lib.oracle_forward.argtypes = [P, P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           P, ctypes.c_int64, P, P]
            lib.oracle_backward.restype = None
            lib.oracle_backward.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int64, P, P, P, P]
            lib.oracle_slot_of_row.restype = ctypes.c_int
            lib.oracle_slot_of_row.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = None
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads(1)
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def build_csr(dst: np.ndarray, N: int):
    """Stable destination CSR: (row_ptr int32 (N+1,), perm int32 (E,), bad count)."""
    dst = _c(dst, np.int32)
    E = dst.shape[0]
    row_ptr = np.zeros(N + 1, np.int32)
    perm = np.zeros(E, np.int32)
    bad = _load().oracle_build_csr(_ptr(dst), E, N, _ptr(row_ptr), _ptr(perm))
    return row_ptr, perm, int(bad)


def ladder(lmax: int):
    """(D, R) of the degree-lmax ladder: D = (lmax+1)^2 node rows, R = D - 1 zonal rows."""
    D = (lmax + 1) ** 2
    return D, D - 1


def _lmax_of(rad) -> int:
    """lmax from the radial operand's slot axis (E, lmax, C)."""
    return int(np.shape(rad)[1]) if np.ndim(rad) == 3 else 3


def forward(coup, rad, row_ptr, perm, N: int, nodes=None):
    """Forward in fp64: (out, absum), each (n_out, D, C); lmax = rad.shape[1]."""
    coup = _c(coup, np.float32)
    rad = _c(rad, np.float32)
    lmax = _lmax_of(rad)
    D, R = ladder(lmax)
    C = rad.shape[2] if rad.ndim == 3 else 0
    row_ptr = _c(row_ptr, np.int32)
    perm = _c(perm, np.int32)
    nodes_a = None if nodes is None else _c(nodes, np.int32)
    n_out = N if nodes_a is None else nodes_a.shape[0]
    out = np.zeros((n_out, D, C), np.float64)
    absum = np.zeros((n_out, D, C), np.float64)
    if n_out and C:
        _load().oracle_forward(_ptr(coup), _ptr(rad), _ptr(row_ptr), _ptr(perm), N, C, lmax,
                               _ptr(nodes_a), 0 if nodes_a is None else n_out,
                               _ptr(out), _ptr(absum))
    return out, absum


def backward(g, coup, rad, dst, N: int, edges=None):
    """Backward in fp64: (d_coup (n, D-1), d_rad (n, lmax, C), abs_dcoup, abs_drad)."""
    g = _c(g, np.float32)
    coup = _c(coup, np.float32)
    rad = _c(rad, np.float32)
    dst = _c(dst, np.int32)
    lmax = _lmax_of(rad)
    D, R = ladder(lmax)
    E = dst.shape[0]
    C = rad.shape[2]
    edges_a = None if edges is None else _c(edges, np.int64)
    n_out = E if edges_a is None else edges_a.shape[0]
    d_coup = np.zeros((n_out, R), np.float64)
    d_rad = np.zeros((n_out, lmax, C), np.float64)
    a_dc = np.zeros((n_out, R), np.float64)
    a_dr = np.zeros((n_out, lmax, C), np.float64)
    if n_out and C:
        _load().oracle_backward(_ptr(g), _ptr(coup), _ptr(rad), _ptr(dst), E, N, C, lmax,
                                _ptr(edges_a), 0 if edges_a is None else n_out,
                                _ptr(d_coup), _ptr(d_rad), _ptr(a_dc), _ptr(a_dr))
    return d_coup, d_rad, a_dc, a_dr


def forward_scaled(coup, rad, row_ptr, perm, N: int, scale):
    """The forward with a per-node factor applied to each node's sum (the degree
    normalisation the pages apply after the operator): (out, absum, out_raw,
    absum_raw), fp64.  Nodes without edges are zero whatever their factor."""
    out_raw, absum_raw = forward(coup, rad, row_ptr, perm, N)
    s = np.asarray(scale, np.float64).reshape(-1)
    rp = np.asarray(row_ptr, np.int64)
    has = (rp[1:] > rp[:-1])[:, None, None]
    with np.errstate(invalid="ignore", over="ignore"):
        out = np.where(has, s[:, None, None] * out_raw, 0.0)
        absum = np.where(has, np.abs(s)[:, None, None] * absum_raw, 0.0)
    return out, absum, out_raw, absum_raw


def backward_scaled(g, coup, rad, dst, N: int, scale, out_raw):
    """Gradients of forward_scaled for the cotangent g of its scaled output:
    (d_coup, d_rad, d_scale, abs_dcoup, abs_drad, abs_dscale), fp64.

    d_coup and d_rad are those of the plain operator times the destination's
    factor (the operator is linear in each node's sum); d_scale[n] is the
    product of g[n] with the node's unscaled sum out_raw[n] over rows 1..D-1."""
    dc, dr, adc, adr = backward(g, coup, rad, dst, N)
    s = np.asarray(scale, np.float64).reshape(-1)
    d = np.asarray(dst, np.int64)
    ok = (d >= 0) & (d < N)
    se = np.where(ok, s[np.where(ok, d, 0)], 0.0)
    with np.errstate(invalid="ignore", over="ignore"):
        dc = dc * se[:, None]
        dr = dr * se[:, None, None]
        adc = adc * np.abs(se)[:, None]
        adr = adr * np.abs(se)[:, None, None]
    g64 = np.asarray(g, np.float64)
    raw = np.asarray(out_raw, np.float64)
    d_scale = np.einsum("nrc,nrc->n", g64[:, 1:], raw[:, 1:])
    abs_ds = np.einsum("nrc,nrc->n", np.abs(g64[:, 1:]), np.abs(raw[:, 1:]))
    return dc, dr, d_scale, adc, adr, abs_ds


def set_threads(n: int) -> None:
    """Threads of the C oracle's node and edge loops (1 by default); results do
    not depend on it (every node's and edge's arithmetic runs on one thread)."""
    _load().oracle_set_threads(int(n))


def slot_of_row(r: int) -> int:
    return int(_load().oracle_slot_of_row(r))


def normalised_error(got, ref, absum):
    """max |got - ref| / absum, with absum == 0 requiring got == 0 exactly.

    Returns (max normalised error, count of nonzero values where absum == 0).
    NaN in got where ref is finite counts as an infinite error.
    """
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    absum = np.asarray(absum, np.float64)
    zero = absum == 0
    bad_zero = int(np.count_nonzero(got[zero] != 0))
    nz = ~zero
    if not np.any(nz):
        return 0.0, bad_zero
    err = np.abs(got[nz] - ref[nz]) / absum[nz]
    err = np.where(np.isnan(err), np.inf, err)
    return float(err.max()), bad_zero
