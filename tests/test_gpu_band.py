"""Coupling rows read from (and their gradient written into) a packed Wigner
band in place: zs_forward_ld / zs_backward_ld on row-strided views, against
the contiguous entry points (bit for bit) and the oracle.

Band reading: per edge a row of 3*D - 2 floats in three segments, the m = 0
segment holding one entry per row of the (D, D) rotation's m = 0 column,
degree 0 first; the zonal coupling is that segment's entries 1..D-1.  The
segment's position in the row is not printed on the pages, so both
placements are tested (offset 0 and after the D - 1 entries of one m = +-1
segment)."""
import numpy as np
import pytest
import torch

import oracle
from equivariant_interatomic_potential_gb300 import workloads, zs
from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu


def _band(w, seg_offset, seed):
    lmax = w.rad.shape[1]
    D = (lmax + 1) ** 2
    rng = np.random.default_rng(seed)
    band = rng.standard_normal((w.E, 3 * D - 2)).astype(np.float32)
    band[:, seg_offset + 1: seg_offset + D] = w.coup
    return band, seg_offset + 1, D


@pytest.mark.parametrize("lmax,C,seg", [(3, 32, 0), (3, 32, 15), (3, 40, 15), (2, 32, 8), (5, 16, 0), (1, 32, 3),
                                        (5, 32, 35)])
def test_band_matches_contiguous_and_oracle(lmax, C, seg):
    w = workloads.make_random(400, 50000, C, seed=lmax * 100 + seg, lmax=lmax, hot_node=2, hot_fraction=0.3)
    band_h, first, D = _band(w, seg, seg + 7)
    band = dev(band_h)
    coup_view = band[:, first:first + D - 1]
    assert coup_view.stride() == (3 * D - 2, 1)
    coup, rad, dst, g = dev(w.coup), dev(w.rad), dev(w.dst), dev(w.grad_out)
    row_ptr, perm, _ = zs.zs_build_csr(dst, w.N)
    out_band = zs.zs_forward_ld(coup_view, rad, row_ptr, perm, w.N)
    out_plain = zs.zs_forward(coup, rad, row_ptr, perm, w.N)
    # the coupling gradient written into a band-shaped buffer, the rest untouched
    grad_band = torch.full((w.E, 3 * D - 2), -7.0, device="cuda")
    dc_view = grad_band[:, first:first + D - 1]
    _, dr_band = zs.zs_backward_ld(g, coup_view, rad, dst, w.N, d_coup=dc_view)
    dc_plain, dr_plain = zs.zs_backward(g, coup, rad, dst, w.N)
    torch.cuda.synchronize()
    zs.zs_check_timeouts()
    assert torch.equal(out_band, out_plain)
    assert torch.equal(dr_band, dr_plain)
    assert torch.equal(dc_view, dc_plain)
    outside = torch.ones_like(grad_band, dtype=torch.bool)
    outside[:, first:first + D - 1] = False
    assert torch.all(grad_band[outside] == -7.0)
    rp, pm, _ = oracle.build_csr(w.dst, w.N)
    ref, absum = oracle.forward(w.coup, w.rad, rp, pm, w.N)
    assert_close(out_band.cpu().numpy(), ref, absum, "forward from the band")
    dc, dr, adc, adr = oracle.backward(w.grad_out, w.coup, w.rad, w.dst, w.N)
    assert_close(dc_view.cpu().numpy(), dc, adc, "d_coup into the band")
    assert_close(dr_band.cpu().numpy(), dr, adr, "d_rad")


def test_ld_argument_checks():
    lib = zs.load()
    fake = 1 << 20
    ws = lib.zs_forward_workspace_bytes(100, 10, 32)
    assert lib.zs_forward_ld(fake, 14, fake, fake, fake, 100, 10, 32, 3, fake, fake, ws, None) == 1
    assert b"stride" in lib.zs_last_error()
    assert lib.zs_backward_ld(fake, fake, 46, fake, fake, 100, 10, 32, 3, fake, 10, fake, None) == 1
    assert b"stride" in lib.zs_last_error()
