"""GPU parity of the split gather, the path small problems take.

When a problem has too few target blocks and source tiles to occupy the
persistent gather, fhd_compute (and the forward pass) evaluate every pair
directly with one target per thread and the sources split into slices across
CTAs, then add the slices' partial rows in a fixed order.  These tests force
that path (fhd_test_set_path) on sizes spanning one and many slices, ragged
target chunks and slices, one source, one target and the single-slice case
that writes the output directly, and compare every output with the fp64
oracle; they also check that the automatic choice takes it for a small
problem and the persistent gather for a large one (bit-identical results to
the forced path), and that it is deterministic.
"""
import numpy as np
import pytest

import oracle
from inputs import make_workload, random_problem
from tests.gpu_helpers import (PATH_AUTO, PATH_PERSISTENT, PATH_SPLIT, PSNR_FAST_DB, TOL_ACCURATE, TOL_FAST,
                               gather_path, gpu_fhd, gpu_fhf, gpu_fwd, psnr_db, rel_l2)

pytestmark = pytest.mark.gpu

ACC, FAST = 0, 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()
    torch.cuda.set_device(0)


def check(got, ref, mode, what):
    err = rel_l2(got, ref)
    if mode == ACC:
        assert err <= TOL_ACCURATE, f"{what}: accurate relL2 {err:.3e}"
    else:
        assert err <= TOL_FAST, f"{what}: fast relL2 {err:.3e}"
        assert psnr_db(got, ref) >= PSNR_FAST_DB, f"{what}: fast PSNR {psnr_db(got, ref):.1f} dB"


# (N, M): one source; fewer sources than one slice; one target over many
# slices; ragged 256-target chunks; many slices of a ragged length; sizes
# where the slice count is capped by the minimum slice length.
SIZES = [(1, 1), (1, 100000), (31, 127), (300, 31), (1000, 129), (2049, 1000), (5000, 3001), (20000, 777),
         (100, 40000)]


@pytest.mark.parametrize("N,M", SIZES)
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_split_fhd(N, M, mode):
    p = random_problem(N, M, kmax=32.0, seed=N + 11 * M)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    with gather_path(PATH_SPLIT):
        check(gpu_fhd(p, mode), ref, mode, f"split F^H D N={N} M={M}")


def test_split_single_slice_writes_output():
    """320000 targets fill more than 8 CTAs per SM with one slice: no partial rows."""
    p = random_problem(320000, 40, kmax=32.0, seed=5)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    with gather_path(PATH_SPLIT):
        check(gpu_fhd(p, ACC), ref, ACC, "split F^H D, one slice")


@pytest.mark.parametrize("N,M", [(1, 1), (127, 31), (3001, 5000), (777, 20000)])
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_split_fwd(N, M, mode):
    p = random_problem(N, M, kmax=32.0, seed=N + 13 * M, op="fwd")
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    with gather_path(PATH_SPLIT):
        check(gpu_fwd(p, mode), ref, mode, f"split F rho N={N} M={M}")


@pytest.mark.parametrize("N,M", [(1, 1), (2500, 700), (4099, 1333)])
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_split_fhf(N, M, mode):
    p = random_problem(N, M, kmax=20.0, seed=N + 17 * M, op="fhf")
    ref = oracle.normal(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    with gather_path(PATH_SPLIT):
        check(gpu_fhf(p, mode), ref, mode, f"split F^H F rho N={N} M={M}")


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_split_workload1(mode):
    p = make_workload(1)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    with gather_path(PATH_SPLIT):
        check(gpu_fhd(p, mode), ref, mode, "split workload 1")


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_automatic_choice(mode):
    """A small problem takes the split gather and a large one the persistent
    gather: the automatic result is bit-identical to the forced path's."""
    small = make_workload(1)
    with gather_path(PATH_AUTO):
        auto_small = gpu_fhd(small, mode)
    with gather_path(PATH_SPLIT):
        split_small = gpu_fhd(small, mode)
    assert np.array_equal(auto_small, split_small)
    large = random_problem(65536, 4096, kmax=32.0, seed=8)
    with gather_path(PATH_AUTO):
        auto_large = gpu_fhd(large, mode)
    with gather_path(PATH_PERSISTENT):
        pers_large = gpu_fhd(large, mode)
    assert np.array_equal(auto_large, pers_large)


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_split_deterministic(mode):
    p = random_problem(3000, 9000, kmax=32.0, seed=31)
    with gather_path(PATH_SPLIT):
        a = gpu_fhd(p, mode)
        b = gpu_fhd(p, mode)
    assert np.array_equal(a, b)

