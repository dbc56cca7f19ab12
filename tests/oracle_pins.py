"""Pins that tie the fp64 oracle to facts outside itself.

Each ``pin_*`` takes an ``oracle.Oracle`` handle and raises AssertionError when
the oracle disagrees with a closed form, a library routine it does not use
(numpy's FFT), an invariant of the operator, or an independent brute-force
evaluation.  ``tests/test_oracle_pins.py`` runs them on the real oracle and
``tests/test_oracle_mutants.py`` checks that every planted mistake trips at
least one of them.

Operators ("Case study - iterative MRI reconstruction", section 17.3, rho_n
equation; section 17.2 for F):
    F^H D : rho_n = sum_m D_m exp(+i 2 pi k_m . x_n)
    F rho : (F rho)_m = sum_n rho_n exp(-i 2 pi k_m . x_n)
"""
from __future__ import annotations

import cmath
import math
import os

import numpy as np

from inputs import grid_coords

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rel(a, b) -> float:
    a, b = np.asarray(a), np.asarray(b)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def load_eighth_roots():
    """Rows of tests/golden/eighth_roots.txt (hand-derived exact values)."""
    rows = []
    with open(os.path.join(GOLDEN, "eighth_roots.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(v) for v in line.split()])
    return np.array(rows)


# ---------------------------------------------------------------- closed forms

def pin_k0_single_sample(orc):
    """One sample at k = 0: exp(0) = 1, so rho_n = D_0 for every voxel, exactly."""
    rng = np.random.default_rng(11)
    x, y, z = (rng.uniform(-0.5, 0.5, 37).astype(np.float32) for _ in range(3))
    D0 = complex(0.75, -1.25)
    rho = orc.adjoint(np.zeros(1), np.zeros(1), np.zeros(1), np.array([D0]), x, y, z)
    assert np.all(rho == D0), rho[:4]


def pin_eighth_roots_adjoint(orc):
    """Single sample, phases at multiples of 1/8 cycle: exact eighth roots of unity.

    Each golden row holds k, x, D and the exact value D*exp(+i 2 pi k.x),
    derived by hand from cos/sin of multiples of pi/4.  Every row uses all
    three coordinates with distinct x, y, z, so a dropped term, a swapped
    coordinate, a wrong sign or a wrong 2 pi shows up.
    """
    g = load_eighth_roots()
    for kx, ky, kz, x, y, z, dr, di, er, ei, fr, fi in g:
        rho = orc.adjoint([kx], [ky], [kz], np.array([complex(dr, di)]), [x], [y], [z])
        assert abs(rho[0] - complex(er, ei)) < 1e-14, (kx, ky, kz, x, y, z, rho[0], er, ei)


def pin_eighth_roots_forward(orc):
    """Single voxel, same table: (F rho)_0 = rho_0 exp(-i 2 pi k.x) (last two golden columns)."""
    g = load_eighth_roots()
    for kx, ky, kz, x, y, z, dr, di, er, ei, fr, fi in g:
        out = orc.forward([x], [y], [z], np.array([complex(dr, di)]), [kx], [ky], [kz])
        assert abs(out[0] - complex(fr, fi)) < 1e-14, (kx, ky, kz, x, y, z, out[0], fr, fi)


# ---------------------------------------------------------------- FFT identities

def _cartesian(n: int, d: int):
    """Voxels on the n^d grid -1/2 + i/n and every integer k in [-n/2, n/2)^d."""
    x, y, z = grid_coords(n, n if d >= 2 else 1, n if d == 3 else 1)
    ks = np.arange(n) - n // 2
    if d == 1:
        kx = ks.astype(np.float64)
        ky = kz = np.zeros_like(kx)
    elif d == 2:
        KY, KX = np.meshgrid(ks, ks, indexing="ij")
        kx, ky, kz = KX.ravel().astype(float), KY.ravel().astype(float), np.zeros(KX.size)
    else:
        KZ, KY, KX = np.meshgrid(ks, ks, ks, indexing="ij")
        kx, ky, kz = KX.ravel().astype(float), KY.ravel().astype(float), KZ.ravel().astype(float)
    return x, y, z, kx, ky, kz


def _to_grid(vals, kx, ky, kz, n, d):
    """Scatter per-k values into an n^d array indexed [kz mod n][ky mod n][kx mod n]."""
    shape = (n,) * d
    A = np.zeros(shape, dtype=np.complex128)
    idx = [kx.astype(int) % n]
    if d >= 2:
        idx.insert(0, ky.astype(int) % n)
    if d == 3:
        idx.insert(0, kz.astype(int) % n)
    A[tuple(idx)] = vals
    return A


def pin_cartesian_adjoint_fft(orc):
    """Integer k on the full Cartesian set: F^H D is an inverse FFT.

    With x_i = -1/2 + i/n: exp(i 2 pi k (-1/2 + i/n)) = (-1)^k exp(i 2 pi k i / n),
    so rho = n^d * ifftn(A) with A[k mod n] = D_k (-1)^(sum k); the array axes
    are (z, y, x) and ravel() gives the x-fastest voxel order.
    """
    rng = np.random.default_rng(5)
    for d, n in ((1, 8), (2, 4), (2, 8), (3, 4)):
        x, y, z, kx, ky, kz = _cartesian(n, d)
        D = rng.standard_normal(kx.size) + 1j * rng.standard_normal(kx.size)
        sign = (-1.0) ** (kx + ky + kz)
        ref = (n ** d) * np.fft.ifftn(_to_grid(D * sign, kx, ky, kz, n, d)).ravel()
        got = orc.adjoint(kx, ky, kz, D, x, y, z)
        assert _rel(got, ref) < 1e-12, (d, n, _rel(got, ref))


def pin_cartesian_forward_fft(orc):
    """Integer k on the full Cartesian set: (F rho)_k = (-1)^(sum k) fftn(rho)[k mod n]."""
    rng = np.random.default_rng(6)
    for d, n in ((1, 8), (2, 4), (3, 4)):
        x, y, z, kx, ky, kz = _cartesian(n, d)
        rho = rng.standard_normal(x.size) + 1j * rng.standard_normal(x.size)
        F = np.fft.fftn(rho.reshape((n,) * d))
        idx = [kx.astype(int) % n]
        if d >= 2:
            idx.insert(0, ky.astype(int) % n)
        if d == 3:
            idx.insert(0, kz.astype(int) % n)
        ref = F[tuple(idx)] * (-1.0) ** (kx + ky + kz)
        got = orc.forward(x, y, z, rho, kx, ky, kz)
        assert _rel(got, ref) < 1e-12, (d, n, _rel(got, ref))


def pin_cartesian_normal_identity(orc):
    """Full Cartesian set: F^H F = n^d I, so the normal operator scales rho by n^d."""
    rng = np.random.default_rng(7)
    for d, n in ((2, 8), (3, 4)):
        x, y, z, kx, ky, kz = _cartesian(n, d)
        rho = rng.standard_normal(x.size) + 1j * rng.standard_normal(x.size)
        got = orc.normal(x, y, z, rho, kx, ky, kz)
        assert _rel(got, (n ** d) * rho) < 1e-12, (d, n)


# ---------------------------------------------------------------- invariants

def pin_hermitian_real(orc):
    """Samples closed under k -> -k with D(-k) = conj D(k): the image is real."""
    rng = np.random.default_rng(8)
    h = rng.uniform(-20, 20, size=(40, 3))
    k = np.concatenate([h, -h])
    Dh = rng.standard_normal(40) + 1j * rng.standard_normal(40)
    D = np.concatenate([Dh, np.conj(Dh)])
    x, y, z = (rng.uniform(-0.5, 0.5, 50) for _ in range(3))
    rho = orc.adjoint(k[:, 0], k[:, 1], k[:, 2], D, x, y, z)
    assert np.max(np.abs(rho.imag)) < 1e-12 * np.max(np.abs(rho.real)), np.max(np.abs(rho.imag))
    assert np.max(np.abs(rho.real)) > 1.0


def pin_linearity(orc):
    """F^H (a D1 + b D2) = a F^H D1 + b F^H D2 for complex a, b."""
    rng = np.random.default_rng(9)
    k = rng.uniform(-10, 10, size=(30, 3))
    x, y, z = (rng.uniform(-0.5, 0.5, 20) for _ in range(3))
    D1 = rng.standard_normal(30) + 1j * rng.standard_normal(30)
    D2 = rng.standard_normal(30) + 1j * rng.standard_normal(30)
    a, b = 0.3 - 1.1j, -2.0 + 0.5j
    lhs = orc.adjoint(k[:, 0], k[:, 1], k[:, 2], a * D1 + b * D2, x, y, z)
    rhs = a * orc.adjoint(k[:, 0], k[:, 1], k[:, 2], D1, x, y, z) + b * orc.adjoint(k[:, 0], k[:, 1], k[:, 2], D2, x, y, z)
    assert _rel(lhs, rhs) < 1e-13


def pin_adjoint_identity(orc):
    """<F rho, D>_M = <rho, F^H D>_N for random non-integer k, rho and D."""
    rng = np.random.default_rng(10)
    k = rng.uniform(-17, 17, size=(45, 3))
    x, y, z = (rng.uniform(-0.5, 0.5, 33) for _ in range(3))
    rho = rng.standard_normal(33) + 1j * rng.standard_normal(33)
    D = rng.standard_normal(45) + 1j * rng.standard_normal(45)
    Frho = orc.forward(x, y, z, rho, k[:, 0], k[:, 1], k[:, 2])
    FhD = orc.adjoint(k[:, 0], k[:, 1], k[:, 2], D, x, y, z)
    lhs = np.vdot(Frho, D)
    rhs = np.vdot(rho, FhD)
    assert abs(lhs - rhs) < 1e-11 * abs(lhs), (lhs, rhs)


def pin_normal_psd(orc):
    """<rho, F^H F rho> = ||F rho||^2: real and non-negative for any k."""
    rng = np.random.default_rng(12)
    k = rng.uniform(-9, 9, size=(25, 3))
    x, y, z = (rng.uniform(-0.5, 0.5, 30) for _ in range(3))
    rho = rng.standard_normal(30) + 1j * rng.standard_normal(30)
    q = np.vdot(rho, orc.normal(x, y, z, rho, k[:, 0], k[:, 1], k[:, 2]))
    Frho = orc.forward(x, y, z, rho, k[:, 0], k[:, 1], k[:, 2])
    assert abs(q.imag) < 1e-11 * abs(q.real)
    assert abs(q.real - np.vdot(Frho, Frho).real) < 1e-11 * abs(q.real)


# ---------------------------------------------------------------- brute force

def pin_bruteforce_4cube(orc):
    """Independent pure-Python evaluation on a 4^3 grid with non-integer k.

    Uses cmath.exp of the unreduced phase and math.fsum per component: a
    different evaluation route from the oracle's reduced-argument sin/cos
    and running double sums.
    """
    rng = np.random.default_rng(13)
    x, y, z = grid_coords(4, 4, 4)
    k = rng.uniform(-6.5, 6.5, size=(17, 3)).astype(np.float32).astype(np.float64)
    D = (rng.standard_normal(17) + 1j * rng.standard_normal(17))
    rho = rng.standard_normal(64) + 1j * rng.standard_normal(64)
    got = orc.adjoint(k[:, 0], k[:, 1], k[:, 2], D, x, y, z)
    gotf = orc.forward(x, y, z, rho, k[:, 0], k[:, 1], k[:, 2])
    X = [(float(a), float(b), float(c)) for a, b, c in zip(x, y, z)]
    K = [tuple(map(float, r)) for r in k]
    for n, (a, b, c) in enumerate(X):
        terms = [complex(D[m]) * cmath.exp(2j * math.pi * (kk[0] * a + kk[1] * b + kk[2] * c)) for m, kk in enumerate(K)]
        ref = complex(math.fsum(t.real for t in terms), math.fsum(t.imag for t in terms))
        assert abs(got[n] - ref) < 1e-12 * max(1.0, abs(ref)), (n, got[n], ref)
    for m, kk in enumerate(K):
        terms = [complex(rho[n]) * cmath.exp(-2j * math.pi * (kk[0] * a + kk[1] * b + kk[2] * c)) for n, (a, b, c) in enumerate(X)]
        ref = complex(math.fsum(t.real for t in terms), math.fsum(t.imag for t in terms))
        assert abs(gotf[m] - ref) < 1e-12 * max(1.0, abs(ref)), (m, gotf[m], ref)


ALL_PINS = [
    pin_k0_single_sample,
    pin_eighth_roots_adjoint,
    pin_eighth_roots_forward,
    pin_cartesian_adjoint_fft,
    pin_cartesian_forward_fft,
    pin_cartesian_normal_identity,
    pin_hermitian_real,
    pin_linearity,
    pin_adjoint_identity,
    pin_normal_psd,
    pin_bruteforce_4cube,
]
