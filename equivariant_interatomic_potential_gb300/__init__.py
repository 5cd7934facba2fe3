"""GB300-native zonal scatter of the geometric initial embedding (lmax = 3).

``libzs`` (C ABI in include/zs.h, CUDA kernels for sm_103a in csrc/) holds the
three steps of the hot path; ``zs`` is its thin Python binding, ``autograd``
the differentiable torch.library operators over it (zs_gie::build_csr,
zs_gie::zonal_scatter), and ``workloads`` draws seeded synthetic graphs.
"""
from . import autograd  # noqa: F401  (registers the zs_gie operators)
from .zs import (  # noqa: F401
    ZsError,
    declared_functions,
    library_path,
    load,
    zs_backward,
    zs_backward_csr,
    zs_check_timeouts,
    zs_build_csr,
    zs_build_csr_workspace_bytes,
    zs_forward,
    zs_forward_workspace_bytes,
)
