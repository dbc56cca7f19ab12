"""The CG oracle against closed forms and a dense solve.

Mutants (planted in the oracle's CG through its test hook): 1 drops the
Tikhonov term, 2 inverts beta.  Each must fail a pin.
"""
import numpy as np
import pytest

import oracle
from inputs import grid_coords
from tests.oracle_pins import _cartesian


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def pin_cartesian_one_step(mutant=0):
    """Full Cartesian set: F^H F = n^d I, so CG stops after one iteration at
    rho = F^H D / (n^d + lam), the inverse DFT of the data when lam = 0."""
    rng = np.random.default_rng(21)
    x, y, z, kx, ky, kz = _cartesian(4, 3)
    D = rng.standard_normal(kx.size) + 1j * rng.standard_normal(kx.size)
    for lam in (0.0, 3.0):
        rho, it, hist = oracle.cg(kx, ky, kz, D, x, y, z, lam=lam, max_iter=5, tol=1e-20, _mutant=mutant)
        b = oracle.adjoint(kx, ky, kz, D, x, y, z)
        assert it == 1 and hist[0] < 1e-20 * np.vdot(b, b).real, (it, hist)
        assert _rel(rho, b / (64 + lam)) < 1e-12


def _dense_normal(kx, ky, kz, x, y, z):
    """A[n, n'] = sum_m exp(i 2 pi k_m . (x_n - x_n')), built with numpy's exp."""
    X = np.stack([x, y, z], 1).astype(np.float64)
    K = np.stack([kx, ky, kz], 1).astype(np.float64)
    E = np.exp(2j * np.pi * (X @ K.T))  # (N, M): exp(i 2 pi k_m . x_n)
    return E @ E.conj().T


def pin_matches_dense_solve(mutant=0):
    """N = 12 voxels, M = 60 random samples: after N iterations CG reaches the
    solution of the dense system (A + lam I) rho = b."""
    rng = np.random.default_rng(22)
    N, M = 12, 60
    x, y, z = (rng.uniform(-0.5, 0.5, N) for _ in range(3))
    k = rng.uniform(-2, 2, size=(M, 3))
    D = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    A = _dense_normal(k[:, 0], k[:, 1], k[:, 2], x, y, z)
    b = oracle.adjoint(k[:, 0], k[:, 1], k[:, 2], D, x, y, z)
    for lam in (0.5, 5.0):
        ref = np.linalg.solve(A + lam * np.eye(N), b)
        rho, it, hist = oracle.cg(k[:, 0], k[:, 1], k[:, 2], D, x, y, z, lam=lam, max_iter=N, _mutant=mutant)
        assert _rel(rho, ref) < 1e-8, (lam, _rel(rho, ref))


def pin_energy_norm_decreases(mutant=0):
    """CG minimises the A-norm of the error over growing Krylov spaces, so it
    never increases from one iteration to the next."""
    rng = np.random.default_rng(23)
    N, M = 10, 50
    x, y, z = (rng.uniform(-0.5, 0.5, N) for _ in range(3))
    k = rng.uniform(-2, 2, size=(M, 3))
    D = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    lam = 1.0
    A = _dense_normal(k[:, 0], k[:, 1], k[:, 2], x, y, z) + lam * np.eye(N)
    b = oracle.adjoint(k[:, 0], k[:, 1], k[:, 2], D, x, y, z)
    ref = np.linalg.solve(A, b)
    last = np.inf
    for it in range(1, N + 1):
        rho, _, _ = oracle.cg(k[:, 0], k[:, 1], k[:, 2], D, x, y, z, lam=lam, max_iter=it, _mutant=mutant)
        e = rho - ref
        en = float(np.vdot(e, A @ e).real)
        assert en <= last * (1 + 1e-9) + 1e-18, (it, en, last)
        last = en


PINS = [pin_cartesian_one_step, pin_matches_dense_solve, pin_energy_norm_decreases]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_cg_pin(pin):
    pin()


@pytest.mark.parametrize("mutant", [1, 2])
def test_cg_mutant_is_caught(mutant):
    caught = 0
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught += 1
    assert caught, f"CG mutant {mutant} passed every pin"
