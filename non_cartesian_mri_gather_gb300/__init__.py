"""Python binding of the fhd C ABI (include/fhd.h): argument marshalling only.

Every step of the computation runs in the CUDA kernels of ``libfhd.so``; this
module turns torch CUDA tensors into pointers, sizes and a stream, allocates
the workspace the library asks for, and raises on a non-OK status.  There is
no CPU path: if the compiled library is missing, importing the binding's
operators raises.

Operators ("Case study - iterative MRI reconstruction", sections 17.2-17.3):

    fhd_compute(k, D, x)     rho_n = sum_m D_m exp(+i 2 pi k_m . x_n)     F^H D
    fwd_compute(x, rho, k)   D_m   = sum_n rho_n exp(-i 2 pi k_m . x_n)   F rho
    fhfrho_apply(x, rho, k)  F^H F rho

Coordinates are passed as three float32 tensors each (x, y, z and kx, ky, kz);
complex data as a (real, imag) pair of float32 tensors.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB, build as build_library

__all__ = [
    "FhdError",
    "MODE_ACCURATE",
    "MODE_FAST",
    "MODE_DIRECT",
    "MODE_ACCURATE_DIRECT",
    "MODE_FAST_DIRECT",
    "OP_FHD",
    "OP_FWD",
    "OP_FHF",
    "load",
    "fhd_compute",
    "fhd_compute_profiled",
    "fwd_compute",
    "fhfrho_apply",
    "fhd_workspace_bytes",
    "fhd_workspace_status",
    "fhd_status_string",
    "fhd_launch_shape",
    "fhd_version",
    "fhd_compute_noalloc",
    "fhd_cg_solve",
    "fhd_compute_variant",
    "VARIANTS",
    "CgWorkspace",
    "Workspace",
]

MODE_ACCURATE = 0
MODE_FAST = 1
MODE_DIRECT = 2  # flag: evaluate every pair directly (no equal-spacing recurrence)
MODE_ACCURATE_DIRECT = 2
MODE_FAST_DIRECT = 3
OP_FHD, OP_FWD, OP_FHF = 0, 1, 2

STATUS_NAMES = {
    0: "FHD_OK",
    1: "FHD_ERR_INVALID_VALUE",
    2: "FHD_ERR_MISALIGNED",
    3: "FHD_ERR_ALIAS",
    4: "FHD_ERR_WORKSPACE",
    5: "FHD_ERR_CUDA",
    6: "FHD_ERR_TIMEOUT",
    7: "FHD_ERR_RANGE",
    8: "FHD_ERR_TOO_LARGE",
}

_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_int = ctypes.c_int

# name -> (restype, argtypes); mirrors include/fhd.h and include/fhd_testing.h
SIGNATURES = {
    "fhd_workspace_bytes": (_sz, [_int, _i64, _i64, _int]),
    "fhd_compute": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _sz, _vp]),
    "fhd_compute_profiled": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _sz,
                                    _vp, _vp, _vp]),
    "fwd_compute": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _sz, _vp]),
    "fhfrho_apply": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp, _sz, _vp]),
    "fhd_workspace_status": (_int, [_vp, _vp]),
    "fhd_status_string": (ctypes.c_char_p, [_int]),
    "fhd_launch_shape": (_int, [_int, _int, _vp, _vp, _vp, _vp, _vp]),
    "fhd_version": (_int, []),
    "fhd_compute_noalloc": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp]),
    "fhd_cg_workspace_bytes": (_sz, [_i64, _i64, _int]),
    "fhd_cg_solve": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, ctypes.c_float, _int,
                            ctypes.c_double, _vp, _vp, _int, _vp, _sz, _vp]),
    "fhd_cg_info": (_int, [_vp, _vp, _vp, _vp, _vp]),
    "fhd_variant_workspace_bytes": (_sz, [_int, _i64, _i64]),
    "fhd_compute_variant": (_int, [_int, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fhd_test_compute_skip_tile": (_int, [_i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _int, _vp,
                                          _sz, _vp, _i64]),
    "fhd_test_schedule": (_int, [_i64, _i64, _int]),
    "fhd_test_set_path": (_int, [_int]),
    "fhd_test_set_step_records": (_int, [_int]),
    "fhd_test_fma2_rate": (_int, [_int, ctypes.POINTER(ctypes.c_double)]),
    "fhd_test_split_shape": (_int, [_i64, _i64, _int, _int, _sz, ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_int64)]),
    "fhd_test_check_array": (_int, [_vp, _sz, _int]),
    "fhd_test_phasor": (_int, [_int, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
}


class FhdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.fhd_status_string(status).decode() if _lib is not None else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libfhd.so (building it first only when asked)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        if not build_if_missing:
            raise ImportError(f"fhd CUDA library not built: {LIB} is missing "
                              "(run `python -m non_cartesian_mri_gather_gb300.build`)")
        build_library()
    lib = ctypes.CDLL(LIB)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise FhdError(status, where)


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


def _stream_ptr(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _n(t) -> int:
    return 0 if t is None else int(t.numel())


def _require(ts, what):
    import torch

    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError(f"{what}: expected contiguous float32 CUDA tensors")


def fhd_workspace_bytes(op: int, N: int, M: int, device: int = 0) -> int:
    return int(load().fhd_workspace_bytes(op, N, M, device))


class Workspace:
    """A device buffer sized by fhd_workspace_bytes, reusable across calls."""

    def __init__(self, op: int, N: int, M: int, device=None):
        import torch

        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.nbytes = fhd_workspace_bytes(op, N, M, dev.index)
        if self.nbytes == 0:
            raise FhdError(1, "fhd_workspace_bytes")
        self.tensor = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()


def _ws(ws, op, N, M, ref):
    if ws is None:
        ws = Workspace(op, N, M, ref.device.index if ref is not None else None)
    return ws


def fhd_compute(kx, ky, kz, Dr, Di, x, y, z, rho_r=None, rho_i=None, mode=MODE_ACCURATE, workspace=None,
                stream=None):
    """rho = F^H D.  Returns (rho_r, rho_i), allocating them when not given."""
    import torch

    lib = load()
    _require((kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i), "fhd_compute")
    N, M = _n(x), _n(kx)
    if rho_r is None:
        rho_r = torch.empty(N, dtype=torch.float32, device=x.device)
    if rho_i is None:
        rho_i = torch.empty(N, dtype=torch.float32, device=x.device)
    ws = _ws(workspace, OP_FHD, N, M, x)
    _check(lib.fhd_compute(M, _ptr(kx), _ptr(ky), _ptr(kz), _ptr(Dr), _ptr(Di), N, _ptr(x), _ptr(y), _ptr(z),
                           _ptr(rho_r), _ptr(rho_i), mode, ws.ptr, ws.nbytes, _stream_ptr(stream)), "fhd_compute")
    return rho_r, rho_i


def _event_handle(ev, stream):
    """cudaEvent_t of a torch.cuda.Event; torch creates the CUDA event lazily on
    its first record(), so an unused event is recorded once to create it."""
    import torch

    if ev.cuda_event == 0:
        ev.record(stream if stream is not None else torch.cuda.current_stream())
    return ev.cuda_event


def fhd_compute_profiled(kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i, mode, workspace, gather_start, gather_stop,
                         stream=None):
    """fhd_compute recording two torch.cuda.Event objects around the gather kernel."""
    lib = load()
    _require((kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i), "fhd_compute_profiled")
    N, M = _n(x), _n(kx)
    e0, e1 = _event_handle(gather_start, stream), _event_handle(gather_stop, stream)
    _check(lib.fhd_compute_profiled(M, _ptr(kx), _ptr(ky), _ptr(kz), _ptr(Dr), _ptr(Di), N, _ptr(x), _ptr(y),
                                    _ptr(z), _ptr(rho_r), _ptr(rho_i), mode, workspace.ptr, workspace.nbytes,
                                    _stream_ptr(stream), e0, e1), "fhd_compute_profiled")
    return rho_r, rho_i


def fwd_compute(x, y, z, rho_r, rho_i, kx, ky, kz, D_r=None, D_i=None, mode=MODE_ACCURATE, workspace=None,
                stream=None):
    """D = F rho.  Returns (D_r, D_i)."""
    import torch

    lib = load()
    _require((x, y, z, rho_r, rho_i, kx, ky, kz, D_r, D_i), "fwd_compute")
    N, M = _n(x), _n(kx)
    if D_r is None:
        D_r = torch.empty(M, dtype=torch.float32, device=kx.device)
    if D_i is None:
        D_i = torch.empty(M, dtype=torch.float32, device=kx.device)
    ws = _ws(workspace, OP_FWD, N, M, kx)
    _check(lib.fwd_compute(N, _ptr(x), _ptr(y), _ptr(z), _ptr(rho_r), _ptr(rho_i), M, _ptr(kx), _ptr(ky), _ptr(kz),
                           _ptr(D_r), _ptr(D_i), mode, ws.ptr, ws.nbytes, _stream_ptr(stream)), "fwd_compute")
    return D_r, D_i


def fhfrho_apply(x, y, z, rho_r, rho_i, kx, ky, kz, out_r=None, out_i=None, mode=MODE_ACCURATE, workspace=None,
                 stream=None):
    """out = F^H F rho.  Returns (out_r, out_i)."""
    import torch

    lib = load()
    _require((x, y, z, rho_r, rho_i, kx, ky, kz, out_r, out_i), "fhfrho_apply")
    N, M = _n(x), _n(kx)
    if out_r is None:
        out_r = torch.empty(N, dtype=torch.float32, device=x.device)
    if out_i is None:
        out_i = torch.empty(N, dtype=torch.float32, device=x.device)
    ws = _ws(workspace, OP_FHF, N, M, x)
    _check(lib.fhfrho_apply(N, _ptr(x), _ptr(y), _ptr(z), _ptr(rho_r), _ptr(rho_i), M, _ptr(kx), _ptr(ky),
                            _ptr(kz), _ptr(out_r), _ptr(out_i), mode, ws.ptr, ws.nbytes, _stream_ptr(stream)),
           "fhfrho_apply")
    return out_r, out_i


def fhd_compute_noalloc(kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i, mode=MODE_ACCURATE, stream=None):
    """rho = F^H D through the entry point that allocates nothing (its scratch is
    a static device array in the library; see fhd_compute_noalloc in fhd.h).
    The outputs must be given: this path allocates no tensors either."""
    lib = load()
    _require((kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i), "fhd_compute_noalloc")
    N, M = _n(x), _n(kx)
    _check(lib.fhd_compute_noalloc(M, _ptr(kx), _ptr(ky), _ptr(kz), _ptr(Dr), _ptr(Di), N, _ptr(x), _ptr(y),
                                   _ptr(z), _ptr(rho_r), _ptr(rho_i), mode, _stream_ptr(stream)),
           "fhd_compute_noalloc")
    return rho_r, rho_i


class CgWorkspace:
    """A device buffer sized by fhd_cg_workspace_bytes, reusable across solves."""

    def __init__(self, N: int, M: int, device=None):
        import torch

        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.nbytes = int(load().fhd_cg_workspace_bytes(N, M, dev.index))
        if self.nbytes == 0:
            raise FhdError(1, "fhd_cg_workspace_bytes")
        self.tensor = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()


def fhd_cg_solve(kx, ky, kz, Dr, Di, x, y, z, lam=0.0, max_iter=10, tol=0.0, rho_r=None, rho_i=None,
                 mode=MODE_ACCURATE, workspace=None, stream=None, info=True):
    """Conjugate gradients on (F^H F + lam I) rho = F^H D (fhd_cg_solve in fhd.h).

    Returns (rho_r, rho_i, info) where info = (iterations, rs_final, stopped)
    read back with fhd_cg_info (a synchronisation), or None when info=False.
    """
    import torch

    lib = load()
    _require((kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i), "fhd_cg_solve")
    N, M = _n(x), _n(kx)
    if rho_r is None:
        rho_r = torch.empty(N, dtype=torch.float32, device=x.device)
    if rho_i is None:
        rho_i = torch.empty(N, dtype=torch.float32, device=x.device)
    ws = workspace if workspace is not None else CgWorkspace(N, M, x.device.index)
    st = _stream_ptr(stream)
    _check(lib.fhd_cg_solve(M, _ptr(kx), _ptr(ky), _ptr(kz), _ptr(Dr), _ptr(Di), N, _ptr(x), _ptr(y), _ptr(z),
                            float(lam), int(max_iter), float(tol), _ptr(rho_r), _ptr(rho_i), mode, ws.ptr,
                            ws.nbytes, st), "fhd_cg_solve")
    if not info:
        return rho_r, rho_i, None
    it, rs, stopped = ctypes.c_int(0), ctypes.c_double(0.0), ctypes.c_int(0)
    _check(lib.fhd_cg_info(ws.ptr, st, ctypes.addressof(it), ctypes.addressof(rs), ctypes.addressof(stopped)),
           "fhd_cg_info")
    return rho_r, rho_i, (it.value, rs.value, stopped.value)


# Comparison kernels of include/fhd_ladder.h: the case study's optimisation
# ladder (L0-L5) and the scatter form.
VARIANTS = {"naive": 0, "fission": 1, "private": 2, "constant": 3, "intrinsics": 4, "unroll": 5, "scatter": 6}


def fhd_compute_variant(variant, kx, ky, kz, Dr, Di, x, y, z, rho_r=None, rho_i=None, workspace=None,
                        stream=None):
    """rho = F^H D with one step of the ladder (`variant`: a VARIANTS key or code)."""
    import torch

    lib = load()
    v = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    _require((kx, ky, kz, Dr, Di, x, y, z, rho_r, rho_i), "fhd_compute_variant")
    N, M = _n(x), _n(kx)
    if rho_r is None:
        rho_r = torch.empty(N, dtype=torch.float32, device=x.device)
    if rho_i is None:
        rho_i = torch.empty(N, dtype=torch.float32, device=x.device)
    if workspace is None:
        nb = int(lib.fhd_variant_workspace_bytes(v, N, M))
        if nb == 0:
            raise FhdError(1, "fhd_variant_workspace_bytes")
        workspace = torch.empty(nb, dtype=torch.uint8, device=x.device)
    _check(lib.fhd_compute_variant(v, M, _ptr(kx), _ptr(ky), _ptr(kz), _ptr(Dr), _ptr(Di), N, _ptr(x), _ptr(y),
                                   _ptr(z), _ptr(rho_r), _ptr(rho_i), workspace.data_ptr(), workspace.numel(),
                                   _stream_ptr(stream)), "fhd_compute_variant")
    return rho_r, rho_i


def fhd_workspace_status(workspace, stream=None) -> int:
    """Synchronise the stream and return the status word as an fhd_status code."""
    return int(load().fhd_workspace_status(workspace.ptr, _stream_ptr(stream)))


def fhd_status_string(status: int) -> str:
    return load().fhd_status_string(status).decode()


def fhd_launch_shape(device: int = 0, mode: int = MODE_FAST) -> dict:
    vals = [ctypes.c_int(0) for _ in range(5)]
    _check(load().fhd_launch_shape(device, mode, *(ctypes.addressof(v) for v in vals)), "fhd_launch_shape")
    keys = ("ctas", "threads", "targets_per_thread", "tile_sources", "stages")
    return {k: v.value for k, v in zip(keys, vals)}


def fhd_version() -> int:
    return int(load().fhd_version())
