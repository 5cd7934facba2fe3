"""libzs builds for sm_103a, loads, exports every declared symbol, and rejects
bad arguments on the host.  No GPU is needed: every call here returns before
any CUDA call is made."""
import ctypes
import os
import subprocess

import pytest

from equivariant_interatomic_potential_gb300 import build, zs

INVALID, UNSUPPORTED = 1, 2


@pytest.fixture(scope="module")
def lib():
    return zs.load()


def test_header_declares_the_boundary():
    names = zs.declared_functions()
    for fn in ("zs_build_csr", "zs_forward", "zs_backward", "zs_backward_csr", "zs_build_csr_workspace_bytes",
               "zs_forward_workspace_bytes", "zs_forward_workspace_bytes_lmax", "zs_status_string", "zs_last_error", "zs_version",
               "zs_check_timeouts", "zs_selftest_bounded_wait", "zs_forward_noalloc", "zs_set_timeout_flag"):
        assert fn in names


def test_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for fn in zs.declared_functions():
        assert fn in exported, fn
        assert getattr(lib, fn) is not None
    # nothing else of ours leaks out of the library
    ours = {s for s in exported if s.startswith("zs_") or "zs" in s.split("_")[0]}
    assert ours <= set(zs.declared_functions())


def test_built_for_sm_103a():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert build.up_to_date()


def test_status_strings(lib):
    assert lib.zs_status_string(0) == b"ZS_OK"
    assert lib.zs_status_string(1) == b"ZS_ERR_INVALID_ARG"
    assert lib.zs_status_string(2) == b"ZS_ERR_UNSUPPORTED"
    assert lib.zs_status_string(3) == b"ZS_ERR_CUDA"
    assert lib.zs_status_string(4) == b"ZS_ERR_TIMEOUT"
    assert lib.zs_status_string(99) == b"ZS_ERR_UNKNOWN"
    assert lib.zs_version() == 10000


FAKE = 1 << 20   # a non-null, 256-byte aligned address never dereferenced by these calls


def test_forward_argument_checks(lib):
    ws = lib.zs_forward_workspace_bytes(100, 10, 32)
    for lmax in (0, 6, -3):   # ladders lmax 1..5 only
        assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, lmax, FAKE, FAKE, 1 << 40, None) == UNSUPPORTED
        assert b"lmax" in lib.zs_last_error()
    # another ladder needs its own, larger workspace
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 5, FAKE, FAKE, ws, None) == INVALID
    assert b"workspace" in lib.zs_last_error()
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, -1, 10, 32, 3, FAKE, FAKE, ws, None) == INVALID
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, -1, 32, 3, FAKE, FAKE, ws, None) == INVALID
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 10, 0, 3, FAKE, FAKE, ws, None) == INVALID
    assert lib.zs_forward(FAKE, FAKE, None, FAKE, 100, 10, 32, 3, FAKE, FAKE, ws, None) == INVALID
    assert lib.zs_forward(None, FAKE, FAKE, FAKE, 100, 10, 32, 3, FAKE, FAKE, ws, None) == INVALID
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 3, None, FAKE, ws, None) == INVALID
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 3, FAKE, FAKE, ws - 1, None) == INVALID
    assert b"workspace" in lib.zs_last_error()
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 3, FAKE, FAKE + 4, ws, None) == INVALID
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 1 << 31, 10, 32, 3, FAKE, FAKE, 1 << 40, None) == INVALID
    # N == 0 is valid and enqueues nothing
    assert lib.zs_forward(FAKE, FAKE, FAKE, FAKE, 100, 0, 32, 3, None, FAKE, ws, None) == 0


def test_backward_argument_checks(lib):
    assert lib.zs_backward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 6, FAKE, FAKE, None) == UNSUPPORTED
    assert lib.zs_backward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 0, FAKE, FAKE, None) == UNSUPPORTED
    assert lib.zs_backward(FAKE, FAKE, FAKE, FAKE, -5, 10, 32, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward(FAKE, FAKE, FAKE, FAKE, 100, 10, -3, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward(FAKE, FAKE, FAKE, None, 100, 10, 32, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward(FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 3, None, FAKE, None) == INVALID
    assert lib.zs_backward(None, FAKE, FAKE, FAKE, 100, 10, 32, 3, FAKE, FAKE, None) == INVALID
    # E == 0 is valid and enqueues nothing
    assert lib.zs_backward(None, None, None, None, 0, 10, 32, 3, None, None, None) == 0


def test_backward_csr_argument_checks(lib):
    assert lib.zs_backward_csr(FAKE, FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 6, FAKE, FAKE, None) == UNSUPPORTED
    assert lib.zs_backward_csr(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 10, 32, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward_csr(FAKE, FAKE, FAKE, None, FAKE, 100, 10, 32, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward_csr(FAKE, FAKE, FAKE, FAKE, None, 100, 10, 32, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward_csr(None, FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 3, FAKE, FAKE, None) == INVALID
    assert lib.zs_backward_csr(FAKE, FAKE, FAKE, FAKE, FAKE, 100, 10, 32, 3, FAKE, None, None) == INVALID
    assert lib.zs_backward_csr(None, None, None, FAKE, None, 0, 10, 32, 3, None, None, None) == 0


def test_selftest_argument_checks(lib):
    assert lib.zs_selftest_bounded_wait(0, None) == INVALID
    assert lib.zs_selftest_bounded_wait((1 << 16) + 1, None) == INVALID


def test_timeout_flag_rejects_memory_the_device_cannot_reach(lib):
    # ordinary (pageable) host memory is not a flag word the kernels may write
    buf = ctypes.create_string_buffer(16)
    assert lib.zs_set_timeout_flag(ctypes.addressof(buf)) == INVALID
    assert b"zs_set_timeout_flag" in lib.zs_last_error()


def test_build_csr_argument_checks(lib):
    ws = lib.zs_build_csr_workspace_bytes(5000, 100)
    assert lib.zs_build_csr(FAKE, -1, 100, FAKE, FAKE, None, FAKE, ws, None) == INVALID
    assert lib.zs_build_csr(FAKE, 5000, -1, FAKE, FAKE, None, FAKE, ws, None) == INVALID
    assert lib.zs_build_csr(FAKE, 5000, 100, None, FAKE, None, FAKE, ws, None) == INVALID
    assert lib.zs_build_csr(None, 5000, 100, FAKE, FAKE, None, FAKE, ws, None) == INVALID
    assert lib.zs_build_csr(FAKE, 5000, 100, FAKE, FAKE, None, FAKE, ws - 1, None) == INVALID
    assert lib.zs_build_csr(FAKE, 5000, 100, FAKE, FAKE, None, FAKE + 8, ws, None) == INVALID
    assert lib.zs_build_csr(FAKE, (1 << 31) - 1, 100, FAKE, FAKE, None, FAKE, 1 << 40, None) == INVALID


def test_workspace_sizes(lib):
    assert lib.zs_build_csr_workspace_bytes(0, 10) == 0
    assert lib.zs_build_csr_workspace_bytes(-1, 10) == 0
    al = lambda x: -(-x // 256) * 256
    # counting path (N + 1 <= 5120): per tile of 512 x rounds edges (rounds so
    # that about 152 tiles cover E, 1..16) one count per key, the key totals,
    # and a 16-bit rank per edge
    def counting(E, N):
        rounds = max(1, min(16, -(-(-(-E // 152)) // 512)))
        T = -(-E // (512 * rounds))
        return al(T * 2 * -(-(N + 1) // 2) * 4) + al((N + 1) * 4) + al(E * 2)
    # radix path: four int32 arrays of E plus a 256 x tiles histogram
    def radix(E):
        return 4 * al(E * 4) + al(256 * -(-E // 2048) * 4) + 1024
    E = 647170
    want = counting(E, 4096)
    for e, n in [(1, 0), (5000, 5119), (2_000_000, 3000), (50, 1)]:
        assert lib.zs_build_csr_workspace_bytes(e, n) == counting(e, n)
    for e, n in [(5000, 5120), (E, 32768), (1, 1 << 20)]:
        assert lib.zs_build_csr_workspace_bytes(e, n) == radix(e)
    assert lib.zs_build_csr_workspace_bytes(E, 4096) == want
    # forward: per window of at least 128 CSR positions (plus one), a pair of 15 x C
    # partials, one crossing-node entry and one 64-bit flag, each array 256-byte aligned
    def ws(E, C):
        w = -(-max(E, 1) // 128) + 1
        return -(-(w * 2 * 15 * C * 4) // 256) * 256 + -(-(w * 4) // 256) * 256 + -(-(w * 8) // 256) * 256
    assert lib.zs_forward_workspace_bytes(E, 4096, 32) == ws(E, 32)
    assert lib.zs_forward_workspace_bytes(0, 4096, 32) == ws(0, 32)
    assert lib.zs_forward_workspace_bytes(1000, 10, 40) == ws(1000, 40)
    # other ladders: the same windows, a pair of R x C partials (R = (lmax+1)^2 - 1),
    # one crossing-node entry and one flag each
    def ws_l(E, C, lmax):
        w = -(-max(E, 1) // 128) + 1
        R = (lmax + 1) ** 2 - 1
        return -(-(w * 2 * R * C * 4) // 256) * 256 + -(-(w * 4) // 256) * 256 + -(-(w * 8) // 256) * 256
    for lmax in (1, 2, 4, 5):
        for e, c in ((E, 32), (0, 7), (1000, 40)):
            assert lib.zs_forward_workspace_bytes_lmax(e, 4096, c, lmax) == ws_l(e, c, lmax)
    assert lib.zs_forward_workspace_bytes_lmax(E, 4096, 32, 3) == ws(E, 32)
    assert lib.zs_forward_workspace_bytes_lmax(E, 4096, 32, 0) == 0
    assert lib.zs_forward_workspace_bytes_lmax(E, 4096, 32, 6) == 0
    assert lib.zs_forward_workspace_bytes(10, 4096, 0) == 0


def test_binding_requires_cuda_tensors():
    import torch
    with pytest.raises(ValueError):
        zs.zs_build_csr(torch.zeros(4, dtype=torch.int32), 3)
