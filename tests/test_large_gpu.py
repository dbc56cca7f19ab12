"""GPU parity past 2^31 voxels: 64-bit target indexing of the persistent gather.

2^31 + 4099 voxels of a 2048 x 1024 x 1025 grid (x fastest; built on the
device, 43 GB with the outputs) and 64 uniform-random samples.  The outputs
at voxels around index 2^31, in the first and last (ragged) target blocks and
at a random spread are compared with the fp64 oracle, and every output must be
finite.  Each thread's 32 voxels lie in one 2048-voxel row, so the gather
takes the equal-spacing recurrence, as on the benchmark grids.
"""
import numpy as np
import pytest

import oracle
from inputs import grid_coords_at, grid_coords_device, uniform_k
from tests.gpu_helpers import TOL_ACCURATE, TOL_FAST, rel_l2

pytestmark = pytest.mark.gpu

NX, NY, NZ = 2048, 1024, 1025
N = 2**31 + 4099
M = 64


@pytest.fixture(scope="module")
def big():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()
    if torch.cuda.get_device_properties(0).total_memory < 64 * 2**30:
        pytest.skip("needs 64 GiB of device memory")
    rng = np.random.default_rng(40)
    kx, ky, kz = uniform_k(rng, M, 32.0)
    Dr = rng.standard_normal(M).astype(np.float32)
    Di = rng.standard_normal(M).astype(np.float32)
    x, y, z = grid_coords_device(N, NX, NY, NZ, "cuda")
    k = [torch.from_numpy(a).cuda() for a in (kx, ky, kz, Dr, Di)]
    yield (kx, ky, kz, Dr, Di), k, (x, y, z)
    del x, y, z
    torch.cuda.empty_cache()


CHUNK = 1 << 28  # finiteness is checked a view of this many elements at a time


def _all_finite(t):
    import torch

    return all(bool(torch.isfinite(t.narrow(0, c0, min(CHUNK, t.numel() - c0))).all())
               for c0 in range(0, t.numel(), CHUNK))


def _indices():
    rng = np.random.default_rng(41)
    edge = [0, 1, 31, 32, 8191, 8192, 2**31 - 8193, 2**31 - 2, 2**31 - 1, 2**31, 2**31 + 1, 2**31 + 4095,
            N - 4099, N - 4098, N - 2, N - 1]
    idx = np.unique(np.concatenate([np.array(edge, dtype=np.int64), rng.integers(0, N, 2000)]))
    assert idx[0] >= 0 and idx[-1] < N  # checked on the host before any device indexing
    return idx


@pytest.mark.parametrize("mode", [0, 1])
def test_fhd_past_2_pow_31_voxels(big, mode):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    (kx, ky, kz, Dr, Di), k, (x, y, z) = big
    rr, ri = fhd.fhd_compute(*k, x, y, z, mode=mode)
    torch.cuda.synchronize()
    assert _all_finite(rr) and _all_finite(ri)
    idx = _indices()
    it = torch.from_numpy(idx).cuda()
    got = (rr[it].double() + 1j * ri[it].double()).cpu().numpy()
    del rr, ri
    ref = oracle.adjoint(kx, ky, kz, Dr + 1j * Di, *grid_coords_at(idx, NX, NY, NZ))
    err = rel_l2(got, ref)
    assert err <= (TOL_ACCURATE if mode == 0 else TOL_FAST), f"relL2 {err:.3e} (mode {mode})"


# ------------------------------------------------------------ many samples

@pytest.mark.parametrize("mode", [0, 1])
def test_split_gather_four_million_samples(mode):
    """256 voxels x 2^22 samples: the split gather with 1216 slices of the
    sample range (the most it uses) against the oracle on every voxel."""
    import non_cartesian_mri_gather_gb300 as fhd
    from inputs import random_problem
    from tests.gpu_helpers import gpu_fhd

    lib = fhd.load()
    p = random_problem(256, 1 << 22, kmax=24.0, seed=42)
    assert lib.fhd_test_split_shape(p.N, p.M, 152, 152, 2 * 152 * 2 * 8192 * 4, None, None) == 1
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    err = rel_l2(gpu_fhd(p, mode), ref)
    assert err <= (TOL_ACCURATE if mode == 0 else TOL_FAST), f"relL2 {err:.3e}"


@pytest.mark.parametrize("mode", [0, 1])
def test_persistent_gather_million_samples(mode):
    """A 64 x 64 x 16 voxel grid x 2^20 samples: 8 target blocks x 4096 sample
    tiles on the persistent gather (every CTA's range splits blocks), checked
    on 512 sampled voxels, first and last included."""
    from inputs import grid_coords, random_problem
    from tests.gpu_helpers import gpu_fhd, sample_indices

    p = random_problem(65536, 1 << 20, kmax=24.0, seed=43)
    p.x, p.y, p.z = grid_coords(64, 64, 16)
    got = gpu_fhd(p, mode)
    idx = np.unique(np.concatenate([[0, p.N - 1], sample_indices(p.N, 512)]))
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x[idx], p.y[idx], p.z[idx])
    err = rel_l2(got[idx], ref)
    assert err <= (TOL_ACCURATE if mode == 0 else TOL_FAST), f"relL2 {err:.3e}"
