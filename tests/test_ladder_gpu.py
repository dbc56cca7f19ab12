"""The comparison kernels of include/fhd_ladder.h against the fp64 oracle.

M = 5000 crosses a 3276-record constant-memory chunk; N = 3000 leaves a
ragged last block.  The variants evaluate sin/cos of the unreduced phase
2 pi k.x in fp32, so k is kept moderate (|k| < 8 cycles/FOV); tolerance
1e-4 for the libm variants and 1e-3 with PSNR >= 60 dB for the hardware
approximations and the scatter form (fp32 atomics in no fixed order).
"""
import numpy as np
import pytest

import oracle
from inputs import random_problem
from tests.gpu_helpers import dev, host_complex, psnr_db, rel_l2

pytestmark = pytest.mark.gpu

LIBM = ["naive", "fission", "private", "constant"]
HW = ["intrinsics", "unroll", "scatter"]


@pytest.fixture(scope="module")
def case():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()
    p = random_problem(3000, 5000, kmax=8.0, seed=41)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    return p, ref


@pytest.mark.parametrize("variant", LIBM + HW)
def test_variant_matches_oracle(case, variant):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    p, ref = case
    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
    rr, ri = fhd.fhd_compute_variant(variant, t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"])
    torch.cuda.synchronize()
    got = host_complex(rr, ri)
    err = rel_l2(got, ref)
    if variant in LIBM:
        assert err <= 1e-4, (variant, err)
    else:
        assert err <= 1e-3 and psnr_db(got, ref) >= 60.0, (variant, err)


def test_variant_rejects_bad_arguments():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    lib = fhd.load()
    d = torch.zeros(16, device="cuda")
    out = [torch.empty(16, device="cuda") for _ in range(2)]
    args = (16, *[d.data_ptr()] * 5, 16, *[d.data_ptr()] * 3, out[0].data_ptr(), out[1].data_ptr())
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    assert lib.fhd_compute_variant(9, *args, ws.data_ptr(), ws.numel(), None) == 1
    assert lib.fhd_compute_variant(1, *args, None, 0, None) == 4  # fission needs its workspace
    bad = (16, *[d.data_ptr()] * 5, 16, *[d.data_ptr()] * 3, d.data_ptr(), out[1].data_ptr())
    assert lib.fhd_compute_variant(2, *bad, ws.data_ptr(), ws.numel(), None) == 3  # output aliases an input
