"""PyTorch operators over libzs, with first-order autograd.

The pull request "fused Triton zonal scatter for the GIE head" (deepmd-kit)
puts the zonal scatter behind a differentiable operator whose backward is
the edge-parallel pass and which has no double backward (sections "What"
and "Tests").  Here that operator is a ``torch.library`` custom op:

  ``zs_gie::build_csr(dst, num_nodes) -> (row_ptr, perm)``
  ``zs_gie::zonal_scatter(coup, rad, dst, row_ptr, perm, num_nodes) -> out``
  ``zs_gie::zonal_scatter_scaled(coup, rad, dst, row_ptr, perm, node_scale,
  num_nodes) -> (out, out_raw)``: the degree normalisation the pages apply
  after the operator (section "What", third bullet), fused: out[n] =
  node_scale[n] * the operator's sum, differentiable in node_scale too

``zonal_scatter``'s backward is ``zs_gie::zonal_scatter_backward``, itself
an operator without a derivative, so a second backward raises.  It takes the
faster of libzs's two backward entry points for the ladder (measured on the
4096-node graph at C = 32): the CSR-order ``zs_backward_csr`` (the forward's
CSR is at hand) at lmax 2, 4 and 5, the edge-order ``zs_backward`` at lmax 1
and 3 and for every other channel count.  Every operator has a fake (meta)
implementation, so ``torch.compile`` traces through them with shapes only;
the launch grid is chosen inside libzs from the runtime sizes.  The
operators run libzs's CUDA kernels and nothing else: CPU tensors are
rejected.  Each call first reads the device's timeout flag (page-locked host
memory, no synchronisation) and raises if a bounded wait of an earlier
launch ran out.
"""
from __future__ import annotations

import torch

from . import zs

_NS = "zs_gie"


def _cuda_only(name: str, *tensors: torch.Tensor) -> None:
    for t in tensors:
        if t.device.type != "cuda":
            raise ValueError(f"{_NS}::{name} runs on CUDA tensors only (got a {t.device.type} tensor)")
    zs.raise_on_timeout_flag(tensors[0].device)


# Ladders whose CSR-order backward is the faster one at C = 32.
CSR_BACKWARD_LADDERS = (2, 4, 5)


def uses_csr_backward(lmax: int, C: int) -> bool:
    """Whether zs_gie::zonal_scatter_backward takes zs_backward_csr for this shape."""
    return C == 32 and lmax in CSR_BACKWARD_LADDERS


@torch.library.custom_op(f"{_NS}::build_csr", mutates_args=())
def build_csr(dst: torch.Tensor, num_nodes: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Stable destination CSR of int32 ``dst``: (row_ptr (N+1,), perm (E,)), int32."""
    _cuda_only("build_csr", dst)
    row_ptr, perm, _ = zs.zs_build_csr(dst.contiguous(), num_nodes)
    return row_ptr, perm


@build_csr.register_fake
def _(dst, num_nodes):
    return (dst.new_empty((num_nodes + 1,), dtype=torch.int32), dst.new_empty(dst.shape, dtype=torch.int32))


@torch.library.custom_op(f"{_NS}::zonal_scatter", mutates_args=())
def zonal_scatter(coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor, row_ptr: torch.Tensor,
                  perm: torch.Tensor, num_nodes: int) -> torch.Tensor:
    """out (N, D, C): row 0 zero, rows 1..D-1 the zonal scatter of coup (E, D-1) x rad (E, lmax, C).

    lmax = rad.shape[1] (3 for the pages' 3/5/7 ladder), D = (lmax + 1)^2."""
    _cuda_only("zonal_scatter", coup, rad, dst, row_ptr, perm)
    return zs.zs_forward(coup.contiguous(), rad.contiguous(), row_ptr.contiguous(), perm.contiguous(), num_nodes)


@zonal_scatter.register_fake
def _(coup, rad, dst, row_ptr, perm, num_nodes):
    # ladder of degree lmax = rad.shape[1]: (lmax + 1)^2 node rows
    return coup.new_empty((num_nodes, (rad.shape[1] + 1) ** 2, rad.shape[2]))


@torch.library.custom_op(f"{_NS}::zonal_scatter_backward", mutates_args=())
def zonal_scatter_backward(grad_out: torch.Tensor, coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor,
                           row_ptr: torch.Tensor, perm: torch.Tensor,
                           num_nodes: int) -> tuple[torch.Tensor, torch.Tensor]:
    """(d_coup (E, D-1), d_rad (E, lmax, C)) for the cotangent grad_out (N, D, C).

    row_ptr and perm are the CSR of dst (the forward's); the ladder and channel
    count pick the entry point (``uses_csr_backward``)."""
    _cuda_only("zonal_scatter_backward", grad_out, coup, rad, dst, row_ptr, perm)
    if uses_csr_backward(rad.shape[1], rad.shape[2]):
        return zs.zs_backward_csr(grad_out.contiguous(), coup.contiguous(), rad.contiguous(), row_ptr.contiguous(),
                                  perm.contiguous(), num_nodes)
    return zs.zs_backward(grad_out.contiguous(), coup.contiguous(), rad.contiguous(), dst.contiguous(), num_nodes)


@zonal_scatter_backward.register_fake
def _(grad_out, coup, rad, dst, row_ptr, perm, num_nodes):
    return coup.new_empty(coup.shape), rad.new_empty(rad.shape)


def _setup_context(ctx, inputs, output):
    coup, rad, dst, row_ptr, perm, num_nodes = inputs
    ctx.save_for_backward(coup, rad, dst, row_ptr, perm)
    ctx.num_nodes = num_nodes


def _backward(ctx, grad_out):
    coup, rad, dst, row_ptr, perm = ctx.saved_tensors
    d_coup, d_rad = zonal_scatter_backward(grad_out, coup, rad, dst, row_ptr, perm, ctx.num_nodes)
    return d_coup, d_rad, None, None, None, None


zonal_scatter.register_autograd(_backward, setup_context=_setup_context)


def zonal_scatter_from_dst(coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor, num_nodes: int) -> torch.Tensor:
    """Build the CSR of dst, then the differentiable zonal scatter."""
    row_ptr, perm = build_csr(dst, num_nodes)
    return zonal_scatter(coup, rad, dst, row_ptr, perm, num_nodes)


@torch.library.custom_op(f"{_NS}::zonal_scatter_scaled", mutates_args=())
def zonal_scatter_scaled(coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor, row_ptr: torch.Tensor,
                         perm: torch.Tensor, node_scale: torch.Tensor,
                         num_nodes: int) -> tuple[torch.Tensor, torch.Tensor]:
    """(out, out_raw): out[n] = node_scale[n] * out_raw[n], out_raw the zonal scatter (N, D, C)."""
    _cuda_only("zonal_scatter_scaled", coup, rad, dst, row_ptr, perm, node_scale)
    return zs.zs_forward_scaled(coup.contiguous(), rad.contiguous(), row_ptr.contiguous(), perm.contiguous(),
                                node_scale.contiguous(), num_nodes)


@zonal_scatter_scaled.register_fake
def _(coup, rad, dst, row_ptr, perm, node_scale, num_nodes):
    shape = (num_nodes, (rad.shape[1] + 1) ** 2, rad.shape[2])
    return coup.new_empty(shape), coup.new_empty(shape)


@torch.library.custom_op(f"{_NS}::zonal_scatter_scaled_backward", mutates_args=())
def zonal_scatter_scaled_backward(grad_out: torch.Tensor, coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor,
                                  node_scale: torch.Tensor, out_raw: torch.Tensor,
                                  num_nodes: int) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(d_coup, d_rad, d_scale) for the cotangent grad_out of the scaled output."""
    _cuda_only("zonal_scatter_scaled_backward", grad_out, coup, rad, dst, node_scale, out_raw)
    return zs.zs_backward_scaled(grad_out.contiguous(), coup.contiguous(), rad.contiguous(), dst.contiguous(),
                                 node_scale.contiguous(), num_nodes, out_raw=out_raw.contiguous())


@zonal_scatter_scaled_backward.register_fake
def _(grad_out, coup, rad, dst, node_scale, out_raw, num_nodes):
    return coup.new_empty(coup.shape), rad.new_empty(rad.shape), node_scale.new_empty(node_scale.shape)


def _setup_context_scaled(ctx, inputs, output):
    coup, rad, dst, row_ptr, perm, node_scale, num_nodes = inputs
    out, out_raw = output
    ctx.mark_non_differentiable(out_raw)
    ctx.save_for_backward(coup, rad, dst, node_scale, out_raw)
    ctx.num_nodes = num_nodes


def _backward_scaled(ctx, grad_out, grad_raw):
    coup, rad, dst, node_scale, out_raw = ctx.saved_tensors
    d_coup, d_rad, d_scale = zonal_scatter_scaled_backward(grad_out, coup, rad, dst, node_scale, out_raw,
                                                           ctx.num_nodes)
    return d_coup, d_rad, None, None, None, d_scale, None


zonal_scatter_scaled.register_autograd(_backward_scaled, setup_context=_setup_context_scaled)


def degree_normalised_scatter(coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor, node_scale: torch.Tensor,
                              num_nodes: int) -> torch.Tensor:
    """CSR of dst, then node_scale[n] * zonal scatter, differentiable in coup, rad and node_scale."""
    row_ptr, perm = build_csr(dst, num_nodes)
    return zonal_scatter_scaled(coup, rad, dst, row_ptr, perm, node_scale, num_nodes)[0]
