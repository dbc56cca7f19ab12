"""The seeded input generators: shapes, determinism and the recipes' stated properties."""
import math
import os

import numpy as np

import inputs
from inputs import (PHANTOM, ellipsoid_image, ellipsoid_kspace, grid_coords, kooshball,
                    make_workload, random_problem, spiral_2d, stack_of_spirals)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_grid_exact_and_x_fastest():
    x, y, z = grid_coords(8, 4, 2)
    assert x.dtype == np.float32 and x.shape == (64,)
    assert np.array_equal(x[:8], (-0.5 + np.arange(8) / 8).astype(np.float32))
    assert np.all(y[:8] == -0.5) and y[8] == -0.25 and z[32] == 0.0 and z[0] == -0.5
    # power-of-two grids are exact in float32
    assert np.array_equal(x.astype(np.float64), -0.5 + (np.arange(64) % 8) / 8)
    x2, y2, z2 = grid_coords(4, 4, 1)
    assert np.all(z2 == 0)


def test_spiral_recipe():
    kx, ky, kz = spiral_2d(4, 512, 16.0, 4.0)
    assert kx.shape == (2048,)
    r = np.hypot(kx.astype(np.float64), ky.astype(np.float64))
    assert r.max() <= 16.0 + 1e-5 and np.all(kz == 0)
    # each interleave starts at the k-space centre
    assert np.all(r[::512] == 0)


def test_stack_of_spirals_recipe():
    kx, ky, kz = stack_of_spirals()
    assert kx.shape == (262144,)
    assert np.array_equal(np.unique(kz), np.arange(-64, 64, 2, dtype=np.float32))
    assert np.hypot(kx, ky).max() <= 64.0 + 1e-4


def test_kooshball_recipe():
    kx, ky, kz = kooshball()
    assert kx.shape == (100000,)
    r = np.sqrt(kx.astype(np.float64) ** 2 + ky.astype(np.float64) ** 2 + kz.astype(np.float64) ** 2)
    assert r.max() <= 128.0 + 1e-3
    # diametral spokes: point 128 of each spoke is the centre
    assert np.all(r[128::256] < 1e-6)


def test_ball_ft_small_q_series_is_continuous():
    q = np.array([0.0, 0.9999e-3, 1.0001e-3])
    B = inputs._unit_ball_ft(q)
    assert abs(B[0] - 4 * math.pi / 3) < 1e-15
    assert abs(B[1] - B[2]) < 1e-8


def test_phantom_dc_equals_volume_integral():
    # F at k = 0 is the integral of the image: sum of A * (4 pi / 3) a b c
    D0 = ellipsoid_kspace(np.zeros(1), np.zeros(1), np.zeros(1))[0]
    ref = sum(A * 4 * math.pi / 3 * ax[0] * ax[1] * ax[2] for _, ax, _, A in PHANTOM)
    assert abs(D0 - ref) < 1e-12


def test_phantom_image_values():
    # the centre lies in the outer shell and the inner body only
    img = ellipsoid_image(np.zeros(1), np.zeros(1), np.zeros(1))
    assert abs(img[0] - (1.0 - 0.6)) < 1e-12
    assert ellipsoid_image(np.array([0.49]), np.zeros(1), np.zeros(1))[0] == 0.0


def test_workloads_deterministic_and_sized():
    for i, (N, M) in ((1, (1024, 2048)), (2, (262144, 16384))):
        a, b = make_workload(i), make_workload(i)
        assert (a.N, a.M) == (N, M)
        for name in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di"):
            assert np.array_equal(getattr(a, name), getattr(b, name)), name
            assert getattr(a, name).dtype == np.float32
    w2 = make_workload(2)
    assert w2.kx.min() >= -32 and w2.kx.max() < 32


def test_random_problem():
    p = random_problem(100, 37, 8.0, seed=3)
    assert p.N == 100 and p.M == 37 and p.Dr.dtype == np.float32
    q = random_problem(100, 37, 8.0, seed=3, op="fhf")
    assert q.rho_r.shape == (100,) and q.pairs == 2 * 100 * 37
    g = random_problem(50, 10, coords="grid")
    assert g.N == 50


def test_page_work_size():
    """The case study's size example: 256^3 voxels x 100k samples is about 1.6e12 pairs,
    and 50 conjugate-gradient iterations about 8e13 (tests/golden/page_sizes.txt)."""
    vals = {}
    with open(os.path.join(GOLDEN, "page_sizes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    pairs = 256 ** 3 * 100000
    assert abs(pairs - vals["pairs_256cube_100k"]) / vals["pairs_256cube_100k"] < 0.05
    assert abs(50 * pairs - vals["pairs_cg50"]) / vals["pairs_cg50"] < 0.05


def test_grid_coords_at_and_device_match_the_grid():
    import torch

    from inputs import grid_coords, grid_coords_at, grid_coords_device

    full = grid_coords(16, 8, 4)
    idx = np.array([0, 1, 15, 16, 127, 128, 511, 300])
    for a, b in zip(grid_coords_at(idx, 16, 8, 4), full):
        assert np.array_equal(a, b[idx])
    dev = grid_coords_device(500, 16, 8, 4, "cpu", chunk=37)
    for a, b in zip(dev, full):
        assert np.array_equal(a.numpy(), b[:500])
    for a, b in zip(grid_coords_device(100, 16, 8, 1, "cpu"), grid_coords(16, 8, 1)):
        assert np.array_equal(a.numpy(), b[:100])
