"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Small problems are compared on every output; they span several target blocks
(8192 targets) and source tiles (256 sources) with ragged tails.  The five
benchmark workloads run at full size in the launch configuration the
benchmark uses; workloads 1-2 are compared on every voxel, workloads 3-4 on a
fixed spread of sampled voxels (a gather output depends only on its own voxel,
so a sampled output is exact for that voxel), and workload 5 through its two
passes plus properties that hold at any size.

Every test here runs the persistent tiled gather (the recurrence paths, the
split target blocks and their fix-up), also on the small sizes the automatic
path choice sends to the split gather; the benchmark workloads run with the
automatic choice, as the benchmark does, and workload 1 also on the persistent
path.  The split gather has its own module (test_split_gpu.py).

Tolerances: relative L2 error <= 1e-5 (accurate mode) and <= 1e-3 with
PSNR >= 60 dB (fast mode).
"""
import numpy as np
import pytest

import oracle
from inputs import make_workload, random_problem
from tests.gpu_helpers import (PATH_AUTO, PATH_PERSISTENT, PSNR_FAST_DB, TOL_ACCURATE, TOL_FAST, gather_path, gpu_fhd,
                               gpu_fhf, gpu_fwd, psnr_db, rel_l2, rel_l2_by_position, sample_indices,
                               step_records)

pytestmark = pytest.mark.gpu

ACC, FAST, ACC_DIRECT, FAST_DIRECT = 0, 1, 2, 3
ALL_MODES = [ACC, FAST, ACC_DIRECT, FAST_DIRECT]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()
    torch.cuda.set_device(0)


@pytest.fixture(autouse=True)
def _persistent_path(request):
    """Persistent gather unless the test asks for the automatic choice."""
    path = PATH_AUTO if "auto_path" in request.keywords else PATH_PERSISTENT
    with gather_path(path):
        yield


def check(got, ref, mode, what):
    err = rel_l2(got, ref)
    if (mode & 1) == 0:
        assert err <= TOL_ACCURATE, f"{what}: accurate relL2 {err:.3e}"
    else:
        assert err <= TOL_FAST, f"{what}: fast relL2 {err:.3e}"
        assert psnr_db(got, ref) >= PSNR_FAST_DB, f"{what}: fast PSNR {psnr_db(got, ref):.1f} dB"
    return err


# ------------------------------------------------------------ small, every output

SIZES = [(1, 1), (31, 127), (1000, 129), (2049, 1000), (5000, 3001), (20000, 777), (100, 40000), (4096, 256)]


@pytest.mark.parametrize("N,M", SIZES)
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fhd_random(N, M, mode):
    p = random_problem(N, M, kmax=32.0, seed=N + 7 * M)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, f"F^H D N={N} M={M}")


@pytest.mark.parametrize("mode", ALL_MODES)
def test_fhd_2d_grid(mode):
    p = random_problem(4500, 1500, kmax=16.0, seed=3, dims=2, coords="grid")
    assert np.all(p.z == 0)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, "F^H D 2D")


@pytest.mark.parametrize("N,M", [(1, 1), (127, 31), (3001, 5000), (777, 20000), (40000, 100)])
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fwd_random(N, M, mode):
    p = random_problem(N, M, kmax=32.0, seed=N + 5 * M, op="fwd")
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    check(gpu_fwd(p, mode), ref, mode, f"F rho N={N} M={M}")


@pytest.mark.parametrize("N,M", [(1, 1), (2500, 700), (4099, 1333)])
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fhf_random(N, M, mode):
    p = random_problem(N, M, kmax=20.0, seed=N + 3 * M, op="fhf")
    ref = oracle.normal(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    check(gpu_fhf(p, mode), ref, mode, f"F^H F rho N={N} M={M}")


# ------------------------------------------------------------ benchmark workloads

_cache = {}


def workload(i):
    if i not in _cache:
        _cache[i] = make_workload(i)
    return _cache[i]


@pytest.mark.parametrize("path", [PATH_AUTO, PATH_PERSISTENT])
@pytest.mark.parametrize("mode", ALL_MODES)
def test_workload1_full(mode, path):
    p = workload(1)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    with gather_path(path):
        check(gpu_fhd(p, mode), ref, mode, f"workload 1 (path {path})")


@pytest.fixture(scope="module")
def ref2():
    p = workload(2)
    return oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)


@pytest.mark.auto_path
@pytest.mark.parametrize("mode", ALL_MODES)
def test_workload2_full(mode, ref2):
    got = gpu_fhd(workload(2), mode)
    check(got, ref2, mode, "workload 2")
    check_by_position(got, ref2, np.arange(got.size), mode, f"workload 2 mode {mode}")


def check_by_position(got, ref, idx, mode, what):
    """The relative L2 error at each position of a thread's 32-target run
    (sampled targets idx), each within the mode's tolerance; prints them."""
    errs = rel_l2_by_position(got, ref, idx)
    worst = max(errs, key=errs.get)
    print(f"{what}: worst position {worst} relL2 {errs[worst]:.3e}; by position "
          + " ".join(f"{q}:{e:.2e}" for q, e in sorted(errs.items())))
    tol = TOL_ACCURATE if (mode & 1) == 0 else TOL_FAST
    assert errs[worst] <= tol, f"{what}: position {worst} relL2 {errs[worst]:.3e}"
    return errs


@pytest.mark.auto_path
@pytest.mark.parametrize("wl", [3, 4])
@pytest.mark.parametrize("mode", ALL_MODES)
def test_workload_sampled(wl, mode):
    """Workloads 3 and 4 on about 4300 voxels: an odd stride meets every
    position of a thread's 32-voxel recurrence run about 134 times, plus the
    edges of three target blocks; each position's relL2 is checked.  The
    pair-by-pair modes (the path of voxels that are not on a grid; the
    benchmark's secondary measurement is accurate mode's) run at full size
    too."""
    p = workload(wl)
    got = gpu_fhd(p, mode)
    idx = sample_indices(p.N, 4096)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x[idx], p.y[idx], p.z[idx])
    check(got[idx], ref, mode, f"workload {wl} ({idx.size} sampled voxels)")
    check_by_position(got[idx], ref, idx, mode, f"workload {wl} mode {mode}")


@pytest.mark.auto_path
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_workload5(mode):
    """F^H F rho at 128^3 x 262144: the forward pass on sampled samples and the
    adjoint pass on sampled voxels against the oracle (the adjoint pass is fed
    the GPU's own float32 F rho, which is exactly what the second pass reads),
    the composed operator equal to fhd_compute(fwd_compute(rho)) bit for bit,
    and <rho, F^H F rho> = ||F rho||^2 (real, positive)."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    from tests.gpu_helpers import dev, host_complex

    p = workload(5)
    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "rho_r", "rho_i")}
    Dr, Di = fhd.fwd_compute(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"], mode=mode)
    o_r, o_i = fhd.fhfrho_apply(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"], mode=mode)
    c_r, c_i = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], Dr, Di, t["x"], t["y"], t["z"], mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(o_r, c_r) and torch.equal(o_i, c_i)
    Frho = host_complex(Dr, Di)
    idx = sample_indices(p.M, 512)
    rho = p.rho_r + 1j * p.rho_i
    ref = oracle.forward(p.x, p.y, p.z, rho, p.kx[idx], p.ky[idx], p.kz[idx])
    check(Frho[idx], ref, mode, "workload 5 forward pass (sampled samples)")
    out = host_complex(o_r, o_i)
    vox = sample_indices(p.N, 4096)
    ref2 = oracle.adjoint(p.kx, p.ky, p.kz, Frho, p.x[vox], p.y[vox], p.z[vox])
    check(out[vox], ref2, mode, f"workload 5 adjoint pass ({vox.size} sampled voxels)")
    check_by_position(out[vox], ref2, vox, mode, f"workload 5 adjoint pass mode {mode}")
    q = np.vdot(rho.astype(np.complex128), out)
    nrm = np.vdot(Frho, Frho).real
    assert abs(q.imag) <= 1e-4 * abs(q.real)
    assert abs(q.real - nrm) <= (1e-4 if mode == ACC else 1e-2) * nrm


# ------------------------------------------------------------ large |k.x|

@pytest.mark.parametrize("kmax", [1024.0, 4096.0])
@pytest.mark.parametrize("coords", ["uniform", "grid"])
@pytest.mark.parametrize("mode", ALL_MODES)
def test_fhd_large_k(kmax, coords, mode):
    """k uniform in [-kmax, kmax)^3 cycles per FOV on a unit FOV, so |k.x|
    reaches about 0.87 kmax cycles (3500 at kmax = 4096), on scattered voxels
    and on a 32^3 grid (the recurrences).  Every sin/cos follows the range
    reduction: fast mode stays within 1e-3 (its float32 phase, one FMA chain,
    carries a rounding error growing with |k.x|: about 6.5e-8 kmax in relative
    L2), accurate mode within 1e-5 (each product reduced on its own)."""
    p = random_problem(32768 if coords == "grid" else 9000, 1500, kmax=kmax, seed=int(kmax) + len(coords),
                       coords=coords)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    err = check(gpu_fhd(p, mode), ref, mode, f"F^H D kmax={kmax:g} {coords}")
    print(f"F^H D kmax={kmax:g} {coords} mode {mode}: relL2 {err:.3e}")


@pytest.mark.parametrize("kmax", [1024.0, 4096.0])
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fwd_large_k(kmax, mode):
    """F rho with the voxels of a 32^3 grid as sources (the source-side
    recurrence) and samples up to kmax cycles per FOV."""
    from inputs import grid_coords

    x, y, z = grid_coords(32, 32, 32)
    p = random_problem(x.size, 1200, kmax=kmax, seed=int(kmax) + 1, op="fwd")
    p.x, p.y, p.z = x, y, z
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    err = check(gpu_fwd(p, mode), ref, mode, f"F rho kmax={kmax:g}")
    print(f"F rho kmax={kmax:g} mode {mode}: relL2 {err:.3e}")


# ------------------------------------------------------------ equal-spacing recurrence

@pytest.mark.parametrize("N,M", [(8197, 1000), (30000, 777), (65536, 300)])
@pytest.mark.parametrize("mode", ALL_MODES)
def test_fhd_3d_grid_ragged(N, M, mode):
    """First N voxels of a 64 x 64 x 16 grid: rows of 64 equally spaced voxels
    (the recurrence runs on 32 per thread), a ragged last row and a ragged last
    block of 8192 targets."""
    from inputs import grid_coords

    gx, gy, gz = grid_coords(64, 64, 16)
    p = random_problem(N, M, kmax=32.0, seed=N + M)
    p.x, p.y, p.z = gx[:N].copy(), gy[:N].copy(), gz[:N].copy()
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, f"F^H D grid N={N} M={M}")


@pytest.mark.parametrize("N,M", [(4096, 1000), (5000, 777)])
@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fhd_small_grid_rows(N, M, mode):
    """16- and 18-wide rows: shorter than a thread's 32 targets, so these warps
    evaluate pair by pair."""
    p = random_problem(N, M, kmax=32.0, seed=N + M, coords="grid")
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, f"F^H D small grid N={N} M={M}")


@pytest.mark.parametrize("mode", ALL_MODES)
def test_rows_with_mixed_spacing(mode):
    """Rows of 32 voxels, each one thread's targets (a warp holds 32 rows).
    Every thread is equally spaced, and the launch's common spacing (that of
    its first two voxels) is 1/32:
    - rows 0-255 alternate between 1/32 and 1/64 every 16 rows, so a warp's
      lanes differ in spacing and each thread evaluates its own step phasor;
    - rows 256-319 (two warps) all have 1/32 and read the step records that
      the pack kernel evaluated for it;
    - rows 320-383 (two warps) all have 1/64: one spacing per warp, but not
      the records' one (the accurate kernel shares one lane's step phasor
      across the warp)."""
    rows = 384
    i = np.arange(32)
    xs = []
    for r in range(rows):
        if r >= 320:
            step = 1 / 64
        else:
            step = 1 / 32 if (r // 16) % 2 == 0 or r >= 256 else 1 / 64
        xs.append(-0.5 + i * step)
    p = random_problem(32 * rows, 900, kmax=16.0, seed=14)
    p.x = np.concatenate(xs).astype(np.float32)
    p.y = np.repeat(((np.arange(rows) % 32) / 32 - 0.5), 32).astype(np.float32)
    p.z = np.repeat(((np.arange(rows) // 32) / 16 - 0.5), 32).astype(np.float32)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, "F^H D mixed row spacing")


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_perturbed_grid_falls_back(mode):
    """One voxel moved by one float32 ulp breaks the exact spacing of its row:
    that warp evaluates pair by pair, the others use the recurrence; all match."""
    p = random_problem(32768, 900, kmax=30.0, seed=5, coords="grid")  # a 32^3 grid
    p.x = p.x.copy()
    p.x[3001] = np.nextafter(p.x[3001], np.float32(1.0))
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, "F^H D perturbed grid")


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_step_records_differ_but_both_match(mode):
    """The adjoint gather's step records (the recurrence's step phasor and
    chain coefficients for the launch's voxel spacing, evaluated once per
    sample in double) against every thread evaluating its own: both match
    the oracle, at every position of a thread's run, and the results are not
    bit-identical, so the records were read."""
    p = random_problem(32768, 2000, kmax=32.0, seed=16, coords="grid")  # a 32^3 grid
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    a = gpu_fhd(p, mode)
    with step_records(0):
        b = gpu_fhd(p, mode)
    tol = TOL_ACCURATE if mode == ACC else TOL_FAST
    for got, what in ((a, "step records"), (b, "per-thread steps")):
        check(got, ref, mode, what)
        worst = max(rel_l2_by_position(got, ref, np.arange(p.N)).values())
        assert worst <= tol, f"{what}: worst position relL2 {worst:.3e}"
    assert not np.array_equal(a, b), "the step records were not used"


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_step_records_for_a_spacing_no_warp_has(mode):
    """A 32^3 grid whose first voxel is moved off the grid: the launch's
    common spacing (that of the first two voxels) is then one no thread has,
    so the step records apply to no warp; the first warp's first thread is
    not equally spaced (that warp evaluates pair by pair) and every other
    warp evaluates its own step phasor.  All match the oracle."""
    p = random_problem(32768, 1500, kmax=30.0, seed=18, coords="grid")
    p.x = p.x.copy()
    p.x[0] = np.float32(-0.4871)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    got = gpu_fhd(p, mode)
    check(got, ref, mode, "F^H D, common spacing of no warp")
    with step_records(0):
        alone = gpu_fhd(p, mode)
    assert np.array_equal(got, alone), "step records were used where no warp has their spacing"


def test_recurrence_and_direct_differ_but_both_match():
    p = random_problem(32768, 2000, kmax=32.0, seed=6, coords="grid")  # a 32^3 grid: exact spacing
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    for fast in (0, 1):
        a = gpu_fhd(p, fast)
        b = gpu_fhd(p, fast | 2)
        check(a, ref, fast, "recurrence")
        check(b, ref, fast | 2, "direct")
        assert not np.array_equal(a, b), "the recurrence path did not run"


@pytest.mark.parametrize("mode", ALL_MODES)
def test_fwd_radial_spokes(mode):
    """F rho with samples along radial spokes: directions rounded to multiples of
    2^-12 make every sample r*d exact in float32, so the samples of a spoke are
    exactly equally spaced targets and take the recurrence."""
    rng = np.random.default_rng(7)
    d = rng.standard_normal((13, 3))
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    d = np.round(d * 4096) / 4096
    r = np.arange(256) - 128.0
    k = (d[:, None, :] * r[None, :, None]).reshape(-1, 3).astype(np.float32)
    assert np.array_equal(k.astype(np.float64), (d[:, None, :] * r[None, :, None]).reshape(-1, 3))
    p = random_problem(3000, k.shape[0], kmax=1.0, seed=7, op="fwd")
    p.kx, p.ky, p.kz = (np.ascontiguousarray(k[:, i]) for i in range(3))
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    check(gpu_fwd(p, mode), ref, mode, "F rho radial")


# ------------------------------------------------------------ source-side recurrence

def _spokes(n_spokes, seed, points=256):
    """Samples along radial spokes whose directions are multiples of 2^-12:
    every sample r*d is exact in float32, so the samples of a spoke are
    exactly equally spaced."""
    rng = np.random.default_rng(seed)
    d = rng.standard_normal((n_spokes, 3))
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    d = np.round(d * 4096) / 4096
    r = np.arange(points) - points / 2
    return (d[:, None, :] * r[None, :, None]).reshape(-1, 3).astype(np.float32)


@pytest.mark.parametrize("side", [32, 24])
@pytest.mark.parametrize("mode", ALL_MODES)
@pytest.mark.parametrize("drop", [0, 5])
def test_fwd_grid_voxel_sources(side, mode, drop):
    """F rho with the voxels of a side^3 grid as sources: rows of 32 are
    equally spaced segments of 32 sources (Clenshaw's recurrence in fast
    mode, Horner's rule in accurate mode); rows of 24 make segments straddle
    rows, so those tiles are evaluated pair by pair.  drop = 5 leaves the last segment with
    fewer real sources than its length (the rest zero-weight padding)."""
    from inputs import grid_coords

    x, y, z = (a[: a.size - drop] for a in grid_coords(side, side, side))
    p = random_problem(x.size, 1500, kmax=side / 2, seed=side, op="fwd")
    p.x, p.y, p.z = x, y, z
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    check(gpu_fwd(p, mode), ref, mode, f"F rho, {side}^3 voxel sources")


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fwd_step_angle_extremes(mode):
    """F rho on a 64^3 grid with samples whose step angle along a voxel row,
    theta = 2 pi k_x / 64, is 0, pi or 2 pi, or just off them: there fast
    mode's Clenshaw recurrence rounds worst (its error grows like eps S^2
    over a segment of S = 32 sources, about 1e-4 relative at worst in a
    float32 emulation), while accurate mode's Horner's rule is unaffected.
    The fast bound here is tighter than the mode's tolerance, so a change
    that makes the recurrence lose more shows."""
    from inputs import grid_coords

    base = np.array([0.0, 32.0, -32.0, 64.0, -64.0])
    kx = np.concatenate([base, base + 1e-3, base - 1e-3, base + 0.01])
    p = random_problem(64 ** 3, kx.size, kmax=32.0, seed=41, op="fwd")
    p.x, p.y, p.z = grid_coords(64, 64, 64)
    p.kx = kx.astype(np.float32)
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    got = gpu_fwd(p, mode)
    check(got, ref, mode, "F rho at step angles 0 and pi")
    if mode == FAST:
        assert rel_l2(got, ref) <= 2e-4, f"fast relL2 {rel_l2(got, ref):.3e}"


@pytest.mark.parametrize("mode", [ACC, FAST])
def test_fwd_perturbed_voxel_sources(mode):
    from inputs import grid_coords

    x, y, z = grid_coords(32, 32, 32)
    x = x.copy()
    x[5000] = np.nextafter(x[5000], np.float32(1.0))  # breaks one segment: its tile goes pair by pair
    p = random_problem(x.size, 1000, kmax=16.0, seed=8, op="fwd")
    p.x, p.y, p.z = x, y, z
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    check(gpu_fwd(p, mode), ref, mode, "F rho, perturbed voxel sources")


def test_source_recurrence_differs_from_direct_but_both_match():
    from inputs import grid_coords

    x, y, z = grid_coords(32, 32, 32)
    p = random_problem(x.size, 2000, kmax=16.0, seed=9, op="fwd")
    p.x, p.y, p.z = x, y, z
    ref = oracle.forward(p.x, p.y, p.z, p.rho_r + 1j * p.rho_i, p.kx, p.ky, p.kz)
    for fast in (0, 1):
        a = gpu_fwd(p, fast)
        b = gpu_fwd(p, fast | 2)
        check(a, ref, fast, "source recurrence")
        check(b, ref, fast | 2, "direct")
        assert not np.array_equal(a, b), "the source recurrence did not run"


@pytest.mark.parametrize("mode", ALL_MODES)
def test_fhd_spoke_sources_random_voxels(mode):
    """F^H D with exactly spaced spoke samples as sources and scattered voxels
    as targets: the source recurrence, not the target one."""
    k = _spokes(11, 10)
    p = random_problem(5000, k.shape[0], kmax=1.0, seed=11)
    p.kx, p.ky, p.kz = (np.ascontiguousarray(k[:, i]) for i in range(3))
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, "F^H D spoke sources")


@pytest.mark.parametrize("mode", ALL_MODES)
def test_source_recurrence_step_changes_within_tile(mode):
    """Spokes of 96 samples (six 16-source segments in fast mode, three
    32-source segments in accurate mode): every 256-source tile holds
    segments of several spokes, so the segment step changes inside a tile
    and the step phasor is re-evaluated there."""
    k = _spokes(23, 12, points=96)
    p = random_problem(4000, k.shape[0], kmax=1.0, seed=12)
    p.kx, p.ky, p.kz = (np.ascontiguousarray(k[:, i]) for i in range(3))
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    check(gpu_fhd(p, mode), ref, mode, "F^H D 96-sample spoke sources")


# ------------------------------------------------------------ polar weights

@pytest.mark.parametrize("coords", ["uniform", "grid"])
@pytest.mark.parametrize("mode", ALL_MODES)
def test_weights_special_values(coords, mode):
    """The adjoint gather stores each weight as {|w|, arg(w) / 2 pi}: exact
    zeros, negative and positive reals (arg = 1/2 and 0 cycles), pure
    imaginary weights (+-1/4), and magnitudes from 1e-30 to 1e30 in one sum,
    all against the oracle."""
    p = random_problem(32768 if coords == "grid" else 5000, 1536, kmax=24.0, seed=90, coords=coords)
    special = np.array([0.0, -1.0, 1.0, 1j, -1j, -0.0, 1e-30, -1e-30j, 2.5 - 0j, -3.0 + 1e-7j], dtype=np.complex128)
    D = (p.Dr + 1j * p.Di).astype(np.complex128)
    D[: special.size * 100] = np.tile(special, 100)
    D[1400:1410] *= 1e30
    p.Dr, p.Di = D.real.astype(np.float32), D.imag.astype(np.float32)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    got = gpu_fhd(p, mode)
    assert np.all(np.isfinite(got))
    check(got, ref, mode, f"F^H D special weights ({coords})")


# ------------------------------------------------------------ edge cases

def test_empty_and_zero_sources():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    d = "cuda"
    x = torch.rand(300, device=d) - 0.5
    e = torch.empty(0, device=d)
    rr, ri = fhd.fhd_compute(e, e, e, e, e, x, x.clone(), x.clone())
    torch.cuda.synchronize()
    assert torch.count_nonzero(rr) == 0 and torch.count_nonzero(ri) == 0
    o_r, o_i = fhd.fhd_compute(x[:5], x[:5].clone(), x[:5].clone(), x[:5].clone(), x[:5].clone(), e, e.clone(),
                               e.clone())
    assert o_r.numel() == 0
    Dr, Di = fhd.fwd_compute(e, e, e, e, e, x, x.clone(), x.clone())
    torch.cuda.synchronize()
    assert torch.count_nonzero(Dr) == 0 and torch.count_nonzero(Di) == 0


@pytest.mark.parametrize("mode", [ACC, FAST])
@pytest.mark.parametrize("coords", ["uniform", "grid"])
def test_deterministic(mode, coords):
    p = random_problem(30000, 5000, kmax=32.0, seed=21, coords=coords)
    a = gpu_fhd(p, mode)
    b = gpu_fhd(p, mode)
    assert np.array_equal(a, b)


def test_workspace_reuse_and_stream():
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    from tests.gpu_helpers import dev, host_complex

    p = random_problem(9000, 2000, kmax=32.0, seed=4)
    ws = fhd.Workspace(fhd.OP_FHF, p.N, p.M)
    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r1 = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"], workspace=ws,
                             stream=s)
        r2 = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"], workspace=ws,
                             stream=s)
    s.synchronize()
    assert fhd.fhd_workspace_status(ws, s) == 0
    a, b = host_complex(*r1), host_complex(*r2)
    assert np.array_equal(a, b)
    ref = oracle.adjoint(p.kx, p.ky, p.kz, p.Dr + 1j * p.Di, p.x, p.y, p.z)
    assert rel_l2(a, ref) <= TOL_ACCURATE
