"""Python binding of libzs (include/zs.h): argument marshalling only.

Every entry point has the name of the C function it calls.  Tensors must be
CUDA tensors of the documented dtype and shape; outputs and workspaces are
allocated with torch when not given.  All compute runs in libzs's kernels;
there is no fallback, and a missing or unbuildable library raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

ZS_OK = 0
STATUS_NAMES = {0: "ZS_OK", 1: "ZS_ERR_INVALID_ARG", 2: "ZS_ERR_UNSUPPORTED", 3: "ZS_ERR_CUDA", 4: "ZS_ERR_TIMEOUT"}


class ZsError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libzs.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libzs.so not found at {_build.LIB}; run equivariant_interatomic_potential_gb300.build")
        lib = ctypes.CDLL(_build.LIB)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.zs_status_string.restype = ctypes.c_char_p
        lib.zs_status_string.argtypes = [ctypes.c_int]
        lib.zs_last_error.restype = ctypes.c_char_p
        lib.zs_last_error.argtypes = []
        lib.zs_version.restype = ctypes.c_int
        lib.zs_version.argtypes = []
        lib.zs_build_csr_workspace_bytes.restype = SZ
        lib.zs_build_csr_workspace_bytes.argtypes = [I64, I32]
        lib.zs_build_csr.restype = ctypes.c_int
        lib.zs_build_csr.argtypes = [P, I64, I32, P, P, P, P, SZ, P]
        lib.zs_forward_workspace_bytes.restype = SZ
        lib.zs_forward_workspace_bytes.argtypes = [I64, I32, I32]
        lib.zs_forward_workspace_bytes_lmax.restype = SZ
        lib.zs_forward_workspace_bytes_lmax.argtypes = [I64, I32, I32, I32]
        lib.zs_forward.restype = ctypes.c_int
        lib.zs_forward.argtypes = [P, P, P, P, I64, I32, I32, I32, P, P, SZ, P]
        lib.zs_backward.restype = ctypes.c_int
        lib.zs_backward.argtypes = [P, P, P, P, I64, I32, I32, I32, P, P, P]
        lib.zs_forward_ld.restype = ctypes.c_int
        lib.zs_forward_ld.argtypes = [P, I64, P, P, P, I64, I32, I32, I32, P, P, SZ, P]
        lib.zs_backward_ld.restype = ctypes.c_int
        lib.zs_backward_ld.argtypes = [P, P, I64, P, P, I64, I32, I32, I32, P, I64, P, P]
        lib.zs_forward_scaled.restype = ctypes.c_int
        lib.zs_forward_scaled.argtypes = [P, P, P, P, P, I64, I32, I32, I32, P, P, P, SZ, P]
        lib.zs_backward_scaled.restype = ctypes.c_int
        lib.zs_backward_scaled.argtypes = [P, P, P, P, P, P, I64, I32, I32, I32, P, P, P, P]
        lib.zs_backward_csr.restype = ctypes.c_int
        lib.zs_backward_csr.argtypes = [P, P, P, P, P, I64, I32, I32, I32, P, P, P]
        lib.zs_forward_noalloc.restype = ctypes.c_int
        lib.zs_forward_noalloc.argtypes = [P, P, P, P, I64, I32, I32, I32, P, P]
        lib.zs_selftest_bounded_wait.restype = ctypes.c_int
        lib.zs_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P]
        lib.zs_check_timeouts.restype = ctypes.c_int
        lib.zs_check_timeouts.argtypes = []
        lib.zs_set_timeout_flag.restype = ctypes.c_int
        lib.zs_set_timeout_flag.argtypes = [P]
        _lib = lib
        return lib


def declared_functions(header: str | None = None) -> list[str]:
    """Names of the functions include/zs.h declares (ZS_API prototypes)."""
    header = header or os.path.join(_build.INCLUDE, "zs.h")
    with open(header) as f:
        text = f.read()
    return re.findall(r"ZS_API\s+[\w\s\*]*?\b(zs_\w+)\s*\(", text)


def _check(fn: str, status: int):
    if status != ZS_OK:
        raise ZsError(fn, status, load().zs_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple):
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_rows(t: torch.Tensor, name: str, shape: tuple) -> int:
    """A float32 CUDA matrix whose rows are contiguous and evenly spaced (a
    view into a wider array allowed): returns the row stride in elements."""
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be torch.float32, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.numel() and (t.stride(1) != 1 or (t.shape[0] > 1 and t.stride(0) < t.shape[1])):
        raise ValueError(f"{name} must have contiguous rows (stride (ld, 1) with ld >= {t.shape[1]})")
    return max(int(t.stride(0)), int(t.shape[1])) if t.shape[0] > 1 else int(t.shape[1])


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def zs_build_csr_workspace_bytes(E: int, N: int) -> int:
    return int(load().zs_build_csr_workspace_bytes(E, N))


def zs_forward_workspace_bytes(E: int, N: int, C: int, lmax: int = 3) -> int:
    return int(load().zs_forward_workspace_bytes_lmax(E, N, C, lmax))


def ladder(lmax: int) -> tuple[int, int]:
    """(D, R): node rows (lmax+1)^2 and zonal rows D - 1 of the degree-lmax ladder."""
    D = (lmax + 1) ** 2
    return D, D - 1


def _lmax(rad: torch.Tensor, lmax: int | None) -> int:
    """The ladder degree: given, else the radial operand's slot count (E, lmax, C)."""
    return int(rad.shape[1]) if lmax is None else int(lmax)


def zs_build_csr(dst: torch.Tensor, N: int, row_ptr=None, perm=None, bad_dst_count=None,
                 workspace=None, stream=None):
    """Stable destination CSR.  Returns (row_ptr (N+1,), perm (E,), bad_dst_count (1,)) int32."""
    E = dst.shape[0]
    dev = dst.device
    _need(dst, "dst", torch.int32, (E,))
    row_ptr = torch.empty(N + 1, dtype=torch.int32, device=dev) if row_ptr is None else row_ptr
    perm = torch.empty(E, dtype=torch.int32, device=dev) if perm is None else perm
    bad_dst_count = torch.empty(1, dtype=torch.int32, device=dev) if bad_dst_count is None else bad_dst_count
    _need(row_ptr, "row_ptr", torch.int32, (N + 1,))
    _need(perm, "perm", torch.int32, (E,))
    need = zs_build_csr_workspace_bytes(E, N)
    if workspace is None:
        workspace = _workspace(need, dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("zs_build_csr", load().zs_build_csr(_ptr(dst), E, N, _ptr(row_ptr), _ptr(perm), _ptr(bad_dst_count),
                                               _ptr(workspace), wbytes, _stream(stream)))
    return row_ptr, perm, bad_dst_count


def zs_forward(coup: torch.Tensor, rad: torch.Tensor, row_ptr: torch.Tensor, perm: torch.Tensor, N: int,
               out=None, workspace=None, stream=None, lmax: int | None = None):
    """Forward zonal scatter.  Returns out (N, D, C) fp32; lmax defaults to rad.shape[1]."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    _need(coup, "coup", torch.float32, (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(row_ptr, "row_ptr", torch.int32, (N + 1,))
    _need(perm, "perm", torch.int32, (E,))
    out = torch.empty((N, D, C), dtype=torch.float32, device=dev) if out is None else out
    _need(out, "out", torch.float32, (N, D, C))
    if workspace is None:
        workspace = _workspace(zs_forward_workspace_bytes(E, N, C, lmax), dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("zs_forward", load().zs_forward(_ptr(coup), _ptr(rad), _ptr(row_ptr), _ptr(perm), E, N, C, lmax,
                                           _ptr(out), _ptr(workspace), wbytes, _stream(stream)))
    return out


def zs_forward_ld(coup: torch.Tensor, rad: torch.Tensor, row_ptr: torch.Tensor, perm: torch.Tensor, N: int,
                  out=None, workspace=None, stream=None, lmax: int | None = None):
    """zs_forward with coup a row-strided view (for example the m = 0 segment of a
    packed (E, 3D-2) Wigner band): coup[e] = coup.data_ptr() + e * coup.stride(0)."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    ld = _need_rows(coup, "coup", (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(row_ptr, "row_ptr", torch.int32, (N + 1,))
    _need(perm, "perm", torch.int32, (E,))
    out = torch.empty((N, D, C), dtype=torch.float32, device=dev) if out is None else out
    _need(out, "out", torch.float32, (N, D, C))
    if workspace is None:
        workspace = _workspace(zs_forward_workspace_bytes(E, N, C, lmax), dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("zs_forward_ld", load().zs_forward_ld(_ptr(coup), ld, _ptr(rad), _ptr(row_ptr), _ptr(perm), E, N, C, lmax,
                                                 _ptr(out), _ptr(workspace), wbytes, _stream(stream)))
    return out


def zs_backward_ld(g: torch.Tensor, coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor, N: int,
                   d_coup: torch.Tensor, d_rad=None, stream=None, lmax: int | None = None):
    """zs_backward with coup and d_coup row-strided views (d_coup must be given)."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    _need(g, "g", torch.float32, (N, D, C))
    ld = _need_rows(coup, "coup", (E, R))
    dld = _need_rows(d_coup, "d_coup", (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(dst, "dst", torch.int32, (E,))
    d_rad = torch.empty((E, lmax, C), dtype=torch.float32, device=dev) if d_rad is None else d_rad
    _need(d_rad, "d_rad", torch.float32, (E, lmax, C))
    _check("zs_backward_ld", load().zs_backward_ld(_ptr(g), _ptr(coup), ld, _ptr(rad), _ptr(dst), E, N, C, lmax,
                                                   _ptr(d_coup), dld, _ptr(d_rad), _stream(stream)))
    return d_coup, d_rad


def zs_forward_scaled(coup: torch.Tensor, rad: torch.Tensor, row_ptr: torch.Tensor, perm: torch.Tensor,
                      node_scale: torch.Tensor, N: int, out=None, out_raw=None, want_raw: bool = True,
                      workspace=None, stream=None, lmax: int | None = None):
    """Forward with the per-node factor fused in.  Returns (out, out_raw); out_raw is
    None when want_raw is False and none is given."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    _need(coup, "coup", torch.float32, (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(row_ptr, "row_ptr", torch.int32, (N + 1,))
    _need(perm, "perm", torch.int32, (E,))
    _need(node_scale, "node_scale", torch.float32, (N,))
    out = torch.empty((N, D, C), dtype=torch.float32, device=dev) if out is None else out
    _need(out, "out", torch.float32, (N, D, C))
    if out_raw is None and want_raw:
        out_raw = torch.empty((N, D, C), dtype=torch.float32, device=dev)
    if out_raw is not None:
        _need(out_raw, "out_raw", torch.float32, (N, D, C))
    if workspace is None:
        workspace = _workspace(zs_forward_workspace_bytes(E, N, C, lmax), dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("zs_forward_scaled", load().zs_forward_scaled(_ptr(coup), _ptr(rad), _ptr(row_ptr), _ptr(perm),
                                                         _ptr(node_scale), E, N, C, lmax, _ptr(out), _ptr(out_raw),
                                                         _ptr(workspace), wbytes, _stream(stream)))
    return out, out_raw


def zs_backward_scaled(g: torch.Tensor, coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor,
                       node_scale: torch.Tensor, N: int, out_raw=None, d_coup=None, d_rad=None, d_scale=None,
                       want_scale_grad: bool = True, stream=None, lmax: int | None = None):
    """Backward of zs_forward_scaled.  Returns (d_coup, d_rad, d_scale); d_scale is
    None unless out_raw is given (and want_scale_grad)."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    _need(g, "g", torch.float32, (N, D, C))
    _need(coup, "coup", torch.float32, (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(dst, "dst", torch.int32, (E,))
    _need(node_scale, "node_scale", torch.float32, (N,))
    d_coup = torch.empty((E, R), dtype=torch.float32, device=dev) if d_coup is None else d_coup
    d_rad = torch.empty((E, lmax, C), dtype=torch.float32, device=dev) if d_rad is None else d_rad
    _need(d_coup, "d_coup", torch.float32, (E, R))
    _need(d_rad, "d_rad", torch.float32, (E, lmax, C))
    if out_raw is not None:
        _need(out_raw, "out_raw", torch.float32, (N, D, C))
        if d_scale is None and want_scale_grad:
            d_scale = torch.empty(N, dtype=torch.float32, device=dev)
    if d_scale is not None:
        _need(d_scale, "d_scale", torch.float32, (N,))
    _check("zs_backward_scaled", load().zs_backward_scaled(_ptr(g), _ptr(coup), _ptr(rad), _ptr(dst),
                                                           _ptr(node_scale), _ptr(out_raw), E, N, C, lmax,
                                                           _ptr(d_coup), _ptr(d_rad), _ptr(d_scale),
                                                           _stream(stream)))
    return d_coup, d_rad, d_scale


def zs_backward(g: torch.Tensor, coup: torch.Tensor, rad: torch.Tensor, dst: torch.Tensor, N: int,
                d_coup=None, d_rad=None, stream=None, lmax: int | None = None):
    """Backward.  Returns (d_coup (E, R), d_rad (E, lmax, C)) fp32; lmax defaults to rad.shape[1]."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    _need(g, "g", torch.float32, (N, D, C))
    _need(coup, "coup", torch.float32, (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(dst, "dst", torch.int32, (E,))
    d_coup = torch.empty((E, R), dtype=torch.float32, device=dev) if d_coup is None else d_coup
    d_rad = torch.empty((E, lmax, C), dtype=torch.float32, device=dev) if d_rad is None else d_rad
    _need(d_coup, "d_coup", torch.float32, (E, R))
    _need(d_rad, "d_rad", torch.float32, (E, lmax, C))
    _check("zs_backward", load().zs_backward(_ptr(g), _ptr(coup), _ptr(rad), _ptr(dst), E, N, C, lmax,
                                             _ptr(d_coup), _ptr(d_rad), _stream(stream)))
    return d_coup, d_rad


def zs_backward_csr(g: torch.Tensor, coup: torch.Tensor, rad: torch.Tensor, row_ptr: torch.Tensor,
                    perm: torch.Tensor, N: int, d_coup=None, d_rad=None, stream=None, lmax: int | None = None):
    """Backward with edges visited in CSR order.  Returns (d_coup (E, R), d_rad (E, lmax, C)) fp32."""
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    dev = coup.device
    _need(g, "g", torch.float32, (N, D, C))
    _need(coup, "coup", torch.float32, (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(row_ptr, "row_ptr", torch.int32, (N + 1,))
    _need(perm, "perm", torch.int32, (E,))
    d_coup = torch.empty((E, R), dtype=torch.float32, device=dev) if d_coup is None else d_coup
    d_rad = torch.empty((E, lmax, C), dtype=torch.float32, device=dev) if d_rad is None else d_rad
    _need(d_coup, "d_coup", torch.float32, (E, R))
    _need(d_rad, "d_rad", torch.float32, (E, lmax, C))
    _check("zs_backward_csr", load().zs_backward_csr(_ptr(g), _ptr(coup), _ptr(rad), _ptr(row_ptr), _ptr(perm),
                                                     E, N, C, lmax, _ptr(d_coup), _ptr(d_rad), _stream(stream)))
    return d_coup, d_rad


def zs_check_timeouts() -> None:
    """Raise ZsError if a bounded device wait ran out since the last check
    (synchronises).  Also clears the current device's page-locked timeout
    flag (``timeout_flag``), if registered: the timeout has been reported."""
    st = load().zs_check_timeouts()
    f = _flags.get(torch.cuda.current_device()) if torch.cuda.is_available() else None
    if f is not None:
        f[0] = 0
    _check("zs_check_timeouts", st)


def zs_set_timeout_flag(flag: torch.Tensor | None) -> None:
    """Register (or, with None, unregister) the current device's timeout flag
    word: an int32 tensor of one element, on the device or in page-locked
    host memory, that the kernels set to 1 when a bounded wait runs out."""
    if flag is not None:
        if flag.dtype != torch.int32 or flag.numel() != 1:
            raise ValueError("the timeout flag is a one-element int32 tensor")
        if flag.device.type == "cpu" and not flag.is_pinned():
            raise ValueError("a host timeout flag must be in page-locked (pinned) memory")
    _check("zs_set_timeout_flag", load().zs_set_timeout_flag(_ptr(flag)))


_flags: dict[int, torch.Tensor] = {}
_flags_lock = threading.Lock()


def _device_index(device) -> int:
    idx = None if device is None else torch.device(device).index
    return torch.cuda.current_device() if idx is None else idx


def timeout_flag(device=None) -> torch.Tensor:
    """The page-locked host word registered for ``device`` (the current CUDA
    device by default), registering it on first use (not during stream
    capture: the registration is a synchronous copy).  It reads 1 once a
    bounded wait of a kernel launched after the registration has run out;
    reading it does not synchronise anything."""
    idx = _device_index(device)
    with _flags_lock:
        f = _flags.get(idx)
        if f is None:
            f = torch.zeros(1, dtype=torch.int32, pin_memory=True)
            with torch.cuda.device(idx):
                zs_set_timeout_flag(f)
            _flags[idx] = f
        return f


def raise_on_timeout_flag(device=None) -> None:
    """Raise ZsError (ZS_ERR_TIMEOUT) if the device's timeout flag is set, and
    clear it.  A host read only: a timeout inside a kernel that has not
    finished yet shows up at a later check.  Registers the flag on first use,
    except while the current stream is being captured."""
    idx = _device_index(device)
    f = _flags.get(idx)
    if f is None:
        if torch.cuda.is_current_stream_capturing():
            return
        f = timeout_flag(idx)
    if int(f[0]) != 0:
        f[0] = 0
        raise ZsError("timeout flag", 4, "a bounded device wait ran out in an earlier launch; its outputs are undefined")


def zs_forward_noalloc(coup: torch.Tensor, rad: torch.Tensor, row_ptr: torch.Tensor, perm: torch.Tensor, N: int,
                       out: torch.Tensor, stream=None, lmax: int | None = None):
    """zs_forward with the library's static device scratch instead of a workspace.

    For callers that cannot allocate device memory: ``out`` must be given,
    nothing is allocated.  See include/zs.h for the size limit and the rule
    that overlapping calls race.
    """
    lmax = _lmax(rad, lmax)
    D, R = ladder(lmax)
    E = coup.shape[0]
    C = rad.shape[2]
    _need(coup, "coup", torch.float32, (E, R))
    _need(rad, "rad", torch.float32, (E, lmax, C))
    _need(row_ptr, "row_ptr", torch.int32, (N + 1,))
    _need(perm, "perm", torch.int32, (E,))
    _need(out, "out", torch.float32, (N, D, C))
    _check("zs_forward_noalloc", load().zs_forward_noalloc(_ptr(coup), _ptr(rad), _ptr(row_ptr), _ptr(perm),
                                                           E, N, C, lmax, _ptr(out), _stream(stream)))
    return out
