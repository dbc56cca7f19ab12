"""fhd_compute_noalloc, the F^H D entry point that allocates nothing.

It serves callers that must not allocate device memory once they are running,
such as a real-time reconstruction loop under a device-memory budget fixed at
start-up, where cudaMalloc could synchronise the device or fail.  Its scratch
is a static device array inside the library, shared by all calls on a device.

The test calls it through the C ABI twice in a row, with different problem
sizes (so the second call runs over the first call's leftovers in the shared
array), and compares each result with the regular fhd_compute, which takes a
caller-allocated workspace, at the tolerances the parity tests use.  It also
checks that a problem above the static limit is refused before any launch.

This file is collected last so that a failure here cannot hide the results of
the other tests in a run that stops at the first failure.
"""
import numpy as np
import pytest

from inputs import random_problem
from tests.gpu_helpers import TOL_ACCURATE, TOL_FAST, dev, host_complex, rel_l2

pytestmark = pytest.mark.gpu

FHD_ERR_TOO_LARGE = 8


@pytest.fixture(scope="module")
def lib():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    torch.cuda.set_device(0)
    return load()


def _noalloc(lib, p, t, out, mode):
    import torch

    st = lib.fhd_compute_noalloc(p.M, t["kx"].data_ptr(), t["ky"].data_ptr(), t["kz"].data_ptr(),
                                 t["Dr"].data_ptr(), t["Di"].data_ptr(), p.N, t["x"].data_ptr(),
                                 t["y"].data_ptr(), t["z"].data_ptr(), out[0].data_ptr(), out[1].data_ptr(), mode,
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("mode", [0, 1])
def test_noalloc_matches_fhd_compute_on_two_calls(lib, mode):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    tol = TOL_ACCURATE if mode == 0 else TOL_FAST
    problems = [random_problem(9000, 5000, kmax=32.0, seed=41), random_problem(3001, 700, kmax=20.0, seed=42)]
    for p in problems:
        t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
        out = [torch.full((p.N,), float("nan"), device="cuda") for _ in range(2)]
        assert _noalloc(lib, p, t, out, mode) == 0
        ref_r, ref_i = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"],
                                       mode=mode)
        torch.cuda.synchronize()
        got, ref = host_complex(*out), host_complex(ref_r, ref_i)
        assert np.all(np.isfinite(got))
        assert rel_l2(got, ref) <= tol, (p.N, p.M, rel_l2(got, ref))


def test_noalloc_refuses_too_many_samples(lib):
    import torch

    big = 131072 + 1  # one sample above the static limit
    d = torch.zeros(big, device="cuda")
    out = [torch.empty(16, device="cuda") for _ in range(2)]
    st = lib.fhd_compute_noalloc(big, *(d.data_ptr() for _ in range(5)), 16, *(d.data_ptr() for _ in range(3)),
                                 out[0].data_ptr(), out[1].data_ptr(), 0, torch.cuda.current_stream().cuda_stream)
    assert st == FHD_ERR_TOO_LARGE


@pytest.mark.parametrize("mode", [0, 1])
def test_noalloc_persistent_path_against_oracle(lib, mode):
    """The persistent gather through the static array: a 64 x 64 x 16 grid with
    16384 samples, then with the maximum 131072 samples (packed records,
    segment descriptors, per-CTA partial slots and their fix-up all in the
    array), and a small problem on the split gather followed by the grid
    again on the same array; every result against the fp64 oracle on sampled
    voxels, and each persistent result bit-identical to fhd_compute."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    import oracle
    from inputs import grid_coords
    from tests.gpu_helpers import sample_indices

    tol = TOL_ACCURATE if mode == 0 else TOL_FAST
    gx, gy, gz = grid_coords(64, 64, 16)

    def grid_problem(M, seed):
        p = random_problem(gx.size, M, kmax=32.0, seed=seed)
        p.x, p.y, p.z = gx.copy(), gy.copy(), gz.copy()
        return p

    calls = [(grid_problem(16384, 43), True), (grid_problem(131072, 44), True),
             (random_problem(3001, 700, kmax=20.0, seed=45), False), (grid_problem(16384, 46), True)]
    for p, persistent in calls:
        # the library's own choice: these grids take the persistent gather,
        # the 3001 x 700 problem the split gather
        t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
        out = [torch.full((p.N,), float("nan"), device="cuda") for _ in range(2)]
        assert _noalloc(lib, p, t, out, mode) == 0
        got = host_complex(*out)
        assert np.all(np.isfinite(got))
        idx = sample_indices(p.N, 2048)
        ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x[idx], p.y[idx], p.z[idx])
        assert rel_l2(got[idx], ref) <= tol, (p.N, p.M, rel_l2(got[idx], ref))
        if persistent:
            ref_r, ref_i = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"],
                                           mode=mode)
            torch.cuda.synchronize()
            assert np.array_equal(got, host_complex(ref_r, ref_i))
