"""Plain fp64 CPU oracle for F^H D, F rho and F^H F rho.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library and
its Python binding never import, link or call it, and there is no CPU
fallback through it.

The arithmetic lives in ``fhd_oracle.c`` (plain C, fp64, OpenMP over the
independent outputs).  This wrapper only promotes float32 arrays to float64
(exact), calls the C routines through ctypes and returns complex128 arrays.

Definitions ("Case study - iterative MRI reconstruction", section 17.3, the
rho_n equation; section 17.2 for the forward operator F):

    adjoint(k, D, x)[n] = sum_m D_m exp(+i 2 pi k_m . x_n)
    forward(x, rho, k)[m] = sum_n rho_n exp(-i 2 pi k_m . x_n)
    normal(x, rho, k) = adjoint(k, forward(x, rho, k), x)   (Fρ kept in fp64)

Every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms,
an FFT identity, Hermitian symmetry, the adjoint identity, brute force), and
``tests/test_oracle_mutants.py`` shows the pins catch planted mistakes.  The
conjugate-gradient loop ``cg`` (plain numpy on these operators) is pinned by
``tests/test_oracle_cg.py``: one-step convergence on a full Cartesian set, a
dense numpy solve, and the monotone energy-norm error.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fhd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict = {}

_D = ctypes.POINTER(ctypes.c_double)


def lib_path(mutant: int = 0) -> str:
    return os.path.join(_BUILD, "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally a planted-mistake variant) with gcc.

    -O2, no -ffast-math, so libm and IEEE double rounding are used as written.
    OpenMP is used when the compiler supports it.
    """
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    if mutant:
        base.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        path = build(mutant)
        self._lib = ctypes.CDLL(path)
        for name in ("oracle_adjoint", "oracle_forward"):
            fn = getattr(self._lib, name)
            fn.restype = None
            fn.argtypes = [ctypes.c_int64, _D, _D, _D, _D, _D, ctypes.c_int64, _D, _D, _D, _D, _D]
        self._lib.oracle_threads.restype = ctypes.c_int
        self._lib.oracle_set_threads.restype = ctypes.c_int
        self._lib.oracle_set_threads.argtypes = [ctypes.c_int]
        self._lib.oracle_mutant_id.restype = ctypes.c_int
        assert self._lib.oracle_mutant_id() == mutant

    @staticmethod
    def _d(a) -> np.ndarray:
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64))

    @staticmethod
    def _p(a: np.ndarray):
        return a.ctypes.data_as(_D)

    def threads(self) -> int:
        return int(self._lib.oracle_threads())

    def set_threads(self, n: int) -> int:
        """Thread count of later calls; returns the previous one."""
        return int(self._lib.oracle_set_threads(int(n)))

    def adjoint(self, kx, ky, kz, D, x, y, z) -> np.ndarray:
        """rho_n = sum_m D_m exp(+i 2 pi k_m . x_n); D complex (or (Dr, Di))."""
        Dr, Di = _split(D)
        kx, ky, kz, Dr, Di = (self._d(a) for a in (kx, ky, kz, Dr, Di))
        x, y, z = (self._d(a) for a in (x, y, z))
        M, N = kx.shape[0], x.shape[0]
        out_r, out_i = np.zeros(N), np.zeros(N)
        self._lib.oracle_adjoint(M, *(self._p(a) for a in (kx, ky, kz, Dr, Di)),
                                 N, *(self._p(a) for a in (x, y, z)), self._p(out_r), self._p(out_i))
        return out_r + 1j * out_i

    def forward(self, x, y, z, rho, kx, ky, kz) -> np.ndarray:
        """(F rho)_m = sum_n rho_n exp(-i 2 pi k_m . x_n); rho complex (or (re, im))."""
        rr, ri = _split(rho)
        x, y, z, rr, ri = (self._d(a) for a in (x, y, z, rr, ri))
        kx, ky, kz = (self._d(a) for a in (kx, ky, kz))
        N, M = x.shape[0], kx.shape[0]
        out_r, out_i = np.zeros(M), np.zeros(M)
        self._lib.oracle_forward(N, *(self._p(a) for a in (x, y, z, rr, ri)),
                                 M, *(self._p(a) for a in (kx, ky, kz)), self._p(out_r), self._p(out_i))
        return out_r + 1j * out_i

    def normal(self, x, y, z, rho, kx, ky, kz, x_out=None, y_out=None, z_out=None) -> np.ndarray:
        """F^H F rho, the forward result kept in fp64.

        ``x_out, y_out, z_out`` optionally restrict the adjoint to a subset of
        voxels (the forward pass always uses every voxel).
        """
        Frho = self.forward(x, y, z, rho, kx, ky, kz)
        if x_out is None:
            x_out, y_out, z_out = x, y, z
        return self.adjoint(kx, ky, kz, Frho, x_out, y_out, z_out)


def _split(v):
    if isinstance(v, tuple):
        return v
    v = np.asarray(v)
    if np.iscomplexobj(v):
        return v.real, v.imag
    return v, np.zeros_like(v, dtype=np.float64)


def get(mutant: int = 0) -> Oracle:
    """Shared handle (built on first use)."""
    with _lock:
        if mutant not in _libs:
            _libs[mutant] = Oracle(mutant)
        return _libs[mutant]


def adjoint(kx, ky, kz, D, x, y, z) -> np.ndarray:
    return get().adjoint(kx, ky, kz, D, x, y, z)


def forward(x, y, z, rho, kx, ky, kz) -> np.ndarray:
    return get().forward(x, y, z, rho, kx, ky, kz)


def normal(x, y, z, rho, kx, ky, kz, **kw) -> np.ndarray:
    return get().normal(x, y, z, rho, kx, ky, kz, **kw)


def cg(kx, ky, kz, D, x, y, z, lam: float = 0.0, max_iter: int = 10, tol: float = 0.0, orc=None,
       _mutant: int = 0):
    """Conjugate gradients on (F^H F + lam I) rho = F^H D, in the order of the
    host loop of "Case study - iterative MRI reconstruction", section 17.3.6:

        b = F^H D;  rho = 0;  r = b;  p = b;  rs_old = <r, r>
        repeat max_iter times:
            Ap = (F^H F + lam I) p
            alpha = rs_old / <p, Ap>
            rho += alpha p;  r -= alpha Ap
            rs_new = <r, r>;  stop if rs_new < tol
            p = r + (rs_new / rs_old) p;  rs_old = rs_new

    (the page's loop has lam = 0; the Tikhonov term lam I is the plainest
    reading of its regulariser R(rho) = ||rho||^2).  <a, b> = sum conj(a) b.
    Returns (rho, iterations, [rs after each iteration]).  `_mutant` plants a
    mistake for the test-suite's mutation checks (0: none).
    """
    orc = orc or get()
    b = orc.adjoint(kx, ky, kz, D, x, y, z)
    rho = np.zeros_like(b)
    r = b.copy()
    p = b.copy()
    rs_old = float(np.vdot(r, r).real)
    hist = []
    it = 0
    for it in range(1, max_iter + 1):
        Ap = orc.normal(x, y, z, p, kx, ky, kz) + (0.0 if _mutant == 1 else lam) * p
        alpha = rs_old / float(np.vdot(p, Ap).real)
        rho = rho + alpha * p
        r = r - alpha * Ap
        rs_new = float(np.vdot(r, r).real)
        hist.append(rs_new)
        if rs_new < tol:
            break
        beta = (rs_old / rs_new) if _mutant == 2 else (rs_new / rs_old)
        p = r + beta * p
        rs_old = rs_new
    return rho, it, hist
