"""Variant B of the oracle: the reference composition.  TEST INFRASTRUCTURE ONLY.

The deepmd-kit pull request "fused Triton zonal scatter for the GIE head",
section "What", describes the eager composition that the fused operator
replaces: broadcast each edge's zonal coupling over its degree's radial rows
(materialising the (E, 15, C) message) and ``index_add_`` it onto the
destination nodes.  This module writes that composition in torch CPU fp64, and
its adjoint (the gradients the composition's autograd would give), so that it
shares no code or loop structure with the C oracle.
"""
from __future__ import annotations

import numpy as np
import torch

# zonal row -> radial slot: degree groups of 2l+1 rows for l = 1..lmax
# (section "Boundary and layout contract": "row groups 3/5/7" at lmax = 3)
ROW_GROUPS = (3, 5, 7)


def row_groups(lmax: int = 3) -> tuple:
    return tuple(2 * l + 1 for l in range(1, lmax + 1))


def slot_index(lmax: int = 3) -> torch.Tensor:
    groups = row_groups(lmax)
    return torch.repeat_interleave(torch.arange(len(groups)), torch.tensor(groups))


def _valid(dst: torch.Tensor, N: int) -> torch.Tensor:
    return (dst >= 0) & (dst < N)


def message(coup, rad) -> torch.Tensor:
    """(E, D-1, C) fp64 message: coupling broadcast over its degree's radial row."""
    coup = torch.as_tensor(np.asarray(coup)).to(torch.float64)
    rad = torch.as_tensor(np.asarray(rad)).to(torch.float64)
    return coup[:, :, None] * rad[:, slot_index(rad.shape[1]), :]


def forward(coup, rad, dst, N: int, chunk: int = 1 << 16) -> np.ndarray:
    """(N, D, C) fp64: scalar row zero, rows 1..D-1 = index_add of the message."""
    coup_t = torch.as_tensor(np.asarray(coup))
    rad_t = torch.as_tensor(np.asarray(rad))
    dst_t = torch.as_tensor(np.asarray(dst)).to(torch.int64)
    E = dst_t.shape[0]
    C = rad_t.shape[2]
    lmax = rad_t.shape[1]
    out = torch.zeros((N, (lmax + 1) ** 2, C), dtype=torch.float64)
    body = out[:, 1:, :]
    for a in range(0, E, chunk):
        b = min(E, a + chunk)
        d = dst_t[a:b]
        keep = _valid(d, N)
        msg = message(coup_t[a:b][keep].numpy(), rad_t[a:b][keep].numpy())
        body.index_add_(0, d[keep], msg)
    return out.numpy()


def backward(g, coup, rad, dst, N: int):
    """Adjoint of the composition: (d_coup (E,D-1), d_rad (E,lmax,C)) in fp64.

    d_msg = g[dst, 1:, :]; d_coup = sum_c d_msg * rad[:, slot(r)];
    d_rad[:, s] = sum over rows r of slot s of d_msg[:, r] * coup[:, r].
    """
    g_t = torch.as_tensor(np.asarray(g)).to(torch.float64)
    coup_t = torch.as_tensor(np.asarray(coup)).to(torch.float64)
    rad_t = torch.as_tensor(np.asarray(rad)).to(torch.float64)
    dst_t = torch.as_tensor(np.asarray(dst)).to(torch.int64)
    E = dst_t.shape[0]
    C = rad_t.shape[2]
    lmax = rad_t.shape[1]
    keep = _valid(dst_t, N)
    d_msg = torch.zeros((E, (lmax + 1) ** 2 - 1, C), dtype=torch.float64)
    d_msg[keep] = g_t[dst_t[keep], 1:, :]
    idx = slot_index(lmax)
    d_coup = (d_msg * rad_t[:, idx, :]).sum(dim=2)
    d_rad = torch.zeros((E, lmax, C), dtype=torch.float64)
    d_rad.index_add_(1, idx, d_msg * coup_t[:, :, None])
    return d_coup.numpy(), d_rad.numpy()


def scaled_with_autograd(coup, rad, dst, N: int, scale, g):
    """The degree-normalised composition with its gradients taken by torch
    autograd in fp64 (no hand-written adjoint): returns (out, d_coup, d_rad,
    d_scale) for the cotangent g of out = scale[n] * composition(n), nodes
    without edges zero."""
    coup_t = torch.as_tensor(np.asarray(coup)).to(torch.float64).requires_grad_(True)
    rad_t = torch.as_tensor(np.asarray(rad)).to(torch.float64).requires_grad_(True)
    s_t = torch.as_tensor(np.asarray(scale)).to(torch.float64).requires_grad_(True)
    dst_t = torch.as_tensor(np.asarray(dst)).to(torch.int64)
    lmax = rad_t.shape[1]
    keep = _valid(dst_t, N)
    msg = coup_t[keep][:, :, None] * rad_t[keep][:, slot_index(lmax), :]
    body = torch.zeros((N, msg.shape[1], rad_t.shape[2]), dtype=torch.float64).index_add(0, dst_t[keep], msg)
    indeg = torch.bincount(dst_t[keep], minlength=N)
    factor = torch.where(indeg > 0, s_t, torch.zeros_like(s_t))
    out = torch.cat([torch.zeros((N, 1, rad_t.shape[2]), dtype=torch.float64), factor[:, None, None] * body], dim=1)
    g_t = torch.as_tensor(np.asarray(g)).to(torch.float64)
    d_coup, d_rad, d_s = torch.autograd.grad(out, (coup_t, rad_t, s_t), g_t)
    return out.detach().numpy(), d_coup.numpy(), d_rad.numpy(), d_s.numpy()
