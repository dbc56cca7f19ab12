"""GPU conjugate gradients (fhd_cg_solve) against the CG oracle.

The oracle runs the same loop in fp64 on the fp64 operators.  The GPU loop
runs the fp32 operators (relative error ~1e-6 accurate, ~1e-5 fast) and fp32
vectors with fp64 dot products, so its iterates drift from the oracle's by
roughly the operator error times the condition number and the iteration
count; with lambda chosen so the system is well conditioned the tests allow
1e-4 (accurate) and 1e-3 (fast) relative L2 difference after 6 iterations.
"""
import numpy as np
import pytest

import oracle
from inputs import random_problem
from tests.gpu_helpers import dev, host_complex, rel_l2
from tests.oracle_pins import _cartesian

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()


def _solve(p, lam, iters, tol=0.0, mode=0, ws=None):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    t = {k: dev(np.asarray(getattr(p, k), dtype=np.float32)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
    rr, ri, info = fhd.fhd_cg_solve(t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"], lam=lam,
                                    max_iter=iters, tol=tol, mode=mode, workspace=ws)
    torch.cuda.synchronize()
    return host_complex(rr, ri), info


class _P:
    pass


def _cart_problem(n=8):
    x, y, z, kx, ky, kz = _cartesian(n, 3)
    rng = np.random.default_rng(31)
    p = _P()
    p.x, p.y, p.z = x, y, z
    p.kx, p.ky, p.kz = (np.asarray(a, np.float32) for a in (kx, ky, kz))
    p.Dr = rng.standard_normal(kx.size).astype(np.float32)
    p.Di = rng.standard_normal(kx.size).astype(np.float32)
    return p


@pytest.mark.parametrize("mode", [0, 1])
def test_cartesian_one_step(mode):
    """Full Cartesian set: F^H F = n^3 I, CG stops after one iteration at b/(n^3 + lam)."""
    p = _cart_problem(8)
    lam = 2.0
    got, (it, rs, stopped) = _solve(p, lam, 5, tol=1e-3, mode=mode)
    ref, oit, _ = oracle.cg(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z, lam=lam, max_iter=5, tol=1e-3)
    assert (it, stopped) == (1, 1) and oit == 1
    assert rel_l2(got, ref) <= (1e-5 if mode == 0 else 1e-3)


@pytest.mark.parametrize("mode", [0, 1])
def test_matches_oracle_cg(mode):
    p = random_problem(4096, 3000, kmax=8.0, seed=32, coords="grid")  # 16^3 grid
    lam = 2000.0
    got, (it, rs, stopped) = _solve(p, lam, 6, mode=mode)
    ref, oit, hist = oracle.cg(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z, lam=lam, max_iter=6)
    assert it == 6 and stopped == 0 and oit == 6
    assert rel_l2(got, ref) <= (1e-4 if mode == 0 else 1e-3), rel_l2(got, ref)
    assert abs(rs - hist[-1]) <= (1e-3 if mode == 0 else 1e-2) * hist[-1]


def test_random_coordinates_direct_path():
    p = random_problem(3000, 2000, kmax=8.0, seed=33)
    lam = 2000.0
    got, _ = _solve(p, lam, 5, mode=0)
    ref, _, _ = oracle.cg(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z, lam=lam, max_iter=5)
    assert rel_l2(got, ref) <= 1e-4


def test_tolerance_stop_and_info():
    p = random_problem(4096, 3000, kmax=8.0, seed=34, coords="grid")
    lam = 2000.0
    ref, oit, hist = oracle.cg(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z, lam=lam, max_iter=50)
    tol = hist[2] * 1.5  # the oracle stops after 3 iterations with this threshold
    ref, oit, _ = oracle.cg(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z, lam=lam, max_iter=50, tol=tol)
    got, (it, rs, stopped) = _solve(p, lam, 50, tol=tol)
    assert oit == 3 and it == 3 and stopped == 1
    assert rel_l2(got, ref) <= 1e-4


def test_deterministic_and_reusable_workspace():
    import non_cartesian_mri_gather_gb300 as fhd

    p = random_problem(4096, 1500, kmax=8.0, seed=35, coords="grid")
    ws = fhd.CgWorkspace(p.N, p.M)
    a, _ = _solve(p, 50.0, 4, ws=ws)
    b, _ = _solve(p, 50.0, 4, ws=ws)
    assert np.array_equal(a, b)


def test_edge_cases():
    p = random_problem(2000, 700, kmax=8.0, seed=36)
    got, (it, rs, stopped) = _solve(p, 1.0, 0)
    assert it == 0 and np.count_nonzero(got) == 0
    q = random_problem(500, 1, kmax=8.0, seed=37)
    q.kx, q.ky, q.kz, q.Dr, q.Di = (np.zeros(0, np.float32) for _ in range(5))
    got, (it, rs, stopped) = _solve(q, 1.0, 3)
    assert np.count_nonzero(got) == 0 and stopped == 1 and it == 0
