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
