"""Seeded synthetic inputs for the non-uniform Fourier sums F^H D and F rho.

This module only *draws* inputs: voxel grids, k-space trajectories, complex
k-space data and complex images.  It holds none of the arithmetic of the
operators themselves (no phase, no sin/cos of k.x, no sum over samples or
voxels), so the CUDA path and the CPU oracle can both consume its arrays
without sharing any of the method.

Sources of the recipes (all synthetic, no dataset):

* "Case study - iterative MRI reconstruction" (brianyu43 PMPP ch.17 notes),
  section 17.1: non-Cartesian trajectories such as spirals and radial
  (kooshball) read-outs; section 17.3: voxel coordinates x_n, sample
  coordinates k_m and data D_m, and the 256^3 voxel x 100k sample example.
* The five benchmark workloads this library is measured on: a 2D 32x32 grid
  with a 4-interleave spiral, a 64^3 grid with uniform random k, a 128^3 grid
  with a stack of spirals and ellipsoid-phantom data, a 256^3 grid with a
  kooshball, and the F^H F operator on the 128^3 stack-of-spirals case.

Units: voxel coordinates are in field-of-view units (the grid spans
[-0.5, 0.5)), k is in cycles per field of view, so the phase of a pair is
2*pi*(k . x) radians.  Every array is returned as contiguous float32, after
being computed in float64.

The ellipsoid phantom's k-space data (workload 3) is the *continuous* Fourier
transform of a sum of ellipsoids, evaluated in closed form (scaling and shift
theorems applied to the transform of a unit ball).  That is data synthesis for
a realistic spectrum, not the discrete sum the library computes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Problem",
    "grid_coords",
    "spiral_2d",
    "uniform_k",
    "stack_of_spirals",
    "kooshball",
    "ellipsoid_kspace",
    "ellipsoid_image",
    "PHANTOM",
    "make_workload",
    "random_problem",
    "WORKLOADS",
]


@dataclass
class Problem:
    """One synthetic problem: voxels x,y,z; samples kx,ky,kz; data.

    For an adjoint problem (F^H D) ``Dr, Di`` hold the k-space data.  For a
    forward / normal-operator problem ``rho_r, rho_i`` hold the image.
    """

    name: str
    x: np.ndarray
    y: np.ndarray
    z: np.ndarray
    kx: np.ndarray
    ky: np.ndarray
    kz: np.ndarray
    Dr: np.ndarray | None = None
    Di: np.ndarray | None = None
    rho_r: np.ndarray | None = None
    rho_i: np.ndarray | None = None
    op: str = "fhd"  # "fhd" (F^H D), "fwd" (F rho) or "fhf" (F^H F rho)
    meta: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return int(self.x.shape[0])

    @property
    def M(self) -> int:
        return int(self.kx.shape[0])

    @property
    def pairs(self) -> int:
        """Voxel-sample pairs one application touches (F^H F counts both passes)."""
        return (2 if self.op == "fhf" else 1) * self.N * self.M


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))


def grid_coords(nx: int, ny: int, nz: int = 1):
    """Regular voxel centres x_i = -0.5 + i/n on each axis, x fastest.

    Linear index n = i + nx*(j + ny*l).  For a 2D grid (nz == 1) z is 0.
    For power-of-two n every coordinate is exact in float32.
    """
    ax = -0.5 + np.arange(nx, dtype=np.float64) / nx
    ay = -0.5 + np.arange(ny, dtype=np.float64) / ny
    az = (-0.5 + np.arange(nz, dtype=np.float64) / nz) if nz > 1 else np.zeros(1)
    z, y, x = np.meshgrid(az, ay, ax, indexing="ij")
    return _f32(x.ravel()), _f32(y.ravel()), _f32(z.ravel())


def grid_coords_at(idx, nx: int, ny: int, nz: int):
    """The coordinates ``grid_coords(nx, ny, nz)`` holds at linear indices
    ``idx`` (int64 array), without building the whole grid."""
    idx = np.asarray(idx, dtype=np.int64)
    x = -0.5 + (idx % nx).astype(np.float64) / nx
    y = -0.5 + ((idx // nx) % ny).astype(np.float64) / ny
    z = (-0.5 + (idx // (nx * ny)).astype(np.float64) / nz) if nz > 1 else np.zeros(idx.shape)
    return _f32(x), _f32(y), _f32(z)


def grid_coords_device(n: int, nx: int, ny: int, nz: int, device, chunk: int = 1 << 26):
    """The first n points of ``grid_coords(nx, ny, nz)`` as float32 torch
    tensors built directly on `device`, a chunk of indices at a time, for
    grids too large to build on the host.  Power-of-two sides keep every
    coordinate exact, equal to ``grid_coords_at``."""
    import torch

    out = [torch.empty(n, dtype=torch.float32, device=device) for _ in range(3)]
    for c0 in range(0, n, chunk):
        i = torch.arange(c0, min(n, c0 + chunk), dtype=torch.int64, device=device)
        out[0][c0:c0 + i.numel()] = (-0.5 + (i % nx).double() / nx).float()
        out[1][c0:c0 + i.numel()] = (-0.5 + ((i // nx) % ny).double() / ny).float()
        out[2][c0:c0 + i.numel()] = ((-0.5 + (i // (nx * ny)).double() / nz).float() if nz > 1
                                     else torch.zeros(i.numel(), device=device))
    return out


def spiral_2d(interleaves: int = 4, points: int = 512, kmax: float = 16.0, turns: float = 4.0):
    """Archimedean multi-interleave spiral in the kx-ky plane (kz = 0).

    Interleave l, point j: t = j/points, r = kmax*t,
    theta = 2*pi*turns*t + 2*pi*l/interleaves; sample index m = points*l + j.
    """
    l = np.repeat(np.arange(interleaves, dtype=np.float64), points)
    j = np.tile(np.arange(points, dtype=np.float64), interleaves)
    t = j / points
    r = kmax * t
    th = 2.0 * math.pi * turns * t + 2.0 * math.pi * l / interleaves
    return _f32(r * np.cos(th)), _f32(r * np.sin(th)), _f32(np.zeros_like(r))


def uniform_k(rng: np.random.Generator, M: int, kmax: float, dims: int = 3):
    """k uniform in [-kmax, kmax)^dims, drawn as one (M, dims) block."""
    k = rng.uniform(-kmax, kmax, size=(M, dims))
    cols = [k[:, d] for d in range(dims)] + [np.zeros(M)] * (3 - dims)
    return tuple(_f32(c) for c in cols)


def stack_of_spirals(planes: int = 64, points: int = 4096, kmax: float = 64.0, turns: float = 64.0):
    """Stack of single-interleave spirals, one per kz plane.

    Plane p has kz = -kmax + 2*kmax*p/planes (64 planes in [-64, 64) by
    default); point j: t = j/points, r = kmax*t, theta = 2*pi*turns*t.
    Sample index m = points*p + j.
    """
    p = np.repeat(np.arange(planes, dtype=np.float64), points)
    j = np.tile(np.arange(points, dtype=np.float64), planes)
    t = j / points
    r = kmax * t
    th = 2.0 * math.pi * turns * t
    kz = -kmax + 2.0 * kmax * p / planes
    return _f32(r * np.cos(th)), _f32(r * np.sin(th)), _f32(kz)


def kooshball(spokes: int = 391, points: int = 256, keep: int = 100000):
    """3D radial (kooshball) trajectory of diametral spokes, |k| <= points/2.

    Spoke s points along a Fibonacci-hemisphere direction
    (z_s = (s + 1/2)/spokes, azimuth s*pi*(3 - sqrt(5))); point j lies at
    radius r_j = j - points/2.  Sample index m = points*s + j; the first
    ``keep`` samples are kept.
    """
    s = np.arange(spokes, dtype=np.float64)
    zs = (s + 0.5) / spokes
    phi = s * math.pi * (3.0 - math.sqrt(5.0))
    rho = np.sqrt(1.0 - zs * zs)
    d = np.stack([rho * np.cos(phi), rho * np.sin(phi), zs], axis=1)  # (spokes, 3)
    r = np.arange(points, dtype=np.float64) - points // 2
    k = (d[:, None, :] * r[None, :, None]).reshape(-1, 3)[:keep]
    return _f32(k[:, 0]), _f32(k[:, 1]), _f32(k[:, 2])


# Ellipsoid phantom: (centre, semi-axes, rotation about z in degrees, intensity).
# A set of our own (no published phantom is implied): an outer shell, an inner
# negative body and three small features.
PHANTOM = (
    ((0.0, 0.0, 0.0), (0.40, 0.30, 0.35), 0.0, 1.0),
    ((0.0, 0.0, 0.0), (0.36, 0.26, 0.31), 0.0, -0.6),
    ((0.12, 0.05, 0.0), (0.08, 0.14, 0.10), 20.0, 0.4),
    ((-0.14, -0.06, 0.05), (0.10, 0.06, 0.12), -15.0, 0.3),
    ((0.0, 0.18, -0.08), (0.05, 0.05, 0.05), 0.0, 0.5),
)


def _rot_z(deg: float) -> np.ndarray:
    a = math.radians(deg)
    c, s = math.cos(a), math.sin(a)
    return np.array([[c, -s, 0.0], [s, c, 0.0], [0.0, 0.0, 1.0]])


def _unit_ball_ft(q: np.ndarray) -> np.ndarray:
    """Continuous FT of the unit-ball indicator at spatial frequency |nu| = q.

    B(q) = (sin(2 pi q) - 2 pi q cos(2 pi q)) / (2 pi^2 q^3), B(0) = 4 pi / 3;
    a short series is used for q < 1e-3 to avoid cancellation.
    """
    q = np.asarray(q, dtype=np.float64)
    out = np.empty_like(q)
    small = q < 1e-3
    a = 2.0 * math.pi * q[~small]
    out[~small] = (np.sin(a) - a * np.cos(a)) / (2.0 * math.pi**2 * q[~small] ** 3)
    a2 = (2.0 * math.pi * q[small]) ** 2
    # sin a - a cos a = a^3/3 - a^5/30 + a^7/840 - ...
    out[small] = (4.0 * math.pi / 3.0) * (1.0 - a2 / 10.0 + a2 * a2 / 280.0)
    return out


def ellipsoid_kspace(kx, ky, kz, phantom=PHANTOM) -> np.ndarray:
    """Closed-form continuous FT (kernel e^{-i 2 pi k.x}) of an ellipsoid sum.

    Ellipsoid {c0 + R diag(a,b,c) u : |u| <= 1} with intensity A transforms
    to A*a*b*c*exp(-i 2 pi k.c0)*B(|diag(a,b,c) R^T k|).  Returns complex128.
    """
    k = np.stack([np.asarray(kx, np.float64), np.asarray(ky, np.float64), np.asarray(kz, np.float64)], axis=1)
    out = np.zeros(k.shape[0], dtype=np.complex128)
    for c0, ax, rot, amp in phantom:
        R = _rot_z(rot)
        kk = (k @ R) * np.asarray(ax)  # rows: diag(ax) R^T k
        q = np.sqrt(np.sum(kk * kk, axis=1))
        shift = np.exp(-2j * math.pi * (k @ np.asarray(c0)))
        out += amp * ax[0] * ax[1] * ax[2] * shift * _unit_ball_ft(q)
    return out


def ellipsoid_image(x, y, z, phantom=PHANTOM) -> np.ndarray:
    """Voxelised phantom: sum of intensities of the ellipsoids containing each voxel centre."""
    p = np.stack([np.asarray(x, np.float64), np.asarray(y, np.float64), np.asarray(z, np.float64)], axis=1)
    img = np.zeros(p.shape[0])
    for c0, ax, rot, amp in phantom:
        R = _rot_z(rot)
        u = ((p - np.asarray(c0)) @ R) / np.asarray(ax)  # R^T (p - c0) scaled
        img += amp * (np.sum(u * u, axis=1) <= 1.0)
    return img


def _workload_1():
    x, y, z = grid_coords(32, 32, 1)
    kx, ky, kz = spiral_2d(4, 512, 16.0, 4.0)
    rng = np.random.default_rng(0)
    Dr, Di = _f32(rng.standard_normal(kx.shape[0])), _f32(rng.standard_normal(kx.shape[0]))
    return Problem("2D 32x32 N=1024, 4-interleave spiral M=2048, F^H D", x, y, z, kx, ky, kz, Dr, Di, op="fhd")


def _workload_2():
    x, y, z = grid_coords(64, 64, 64)
    rng = np.random.default_rng(1)
    kx, ky, kz = uniform_k(rng, 16384, 32.0, 3)
    Dr, Di = _f32(rng.standard_normal(16384)), _f32(rng.standard_normal(16384))
    return Problem("3D 64^3 N=262144, uniform k M=16384, F^H D", x, y, z, kx, ky, kz, Dr, Di, op="fhd")


def _workload_3():
    x, y, z = grid_coords(128, 128, 128)
    kx, ky, kz = stack_of_spirals(64, 4096, 64.0, 64.0)
    rng = np.random.default_rng(2)
    D = ellipsoid_kspace(kx, ky, kz)
    sigma = 0.01 * float(np.max(np.abs(D)))
    M = kx.shape[0]
    D = D + sigma * (rng.standard_normal(M) + 1j * rng.standard_normal(M))
    return Problem("3D 128^3 N=2097152, stack of spirals M=262144, phantom data, F^H D",
                   x, y, z, kx, ky, kz, _f32(D.real), _f32(D.imag), op="fhd")


def _workload_4():
    x, y, z = grid_coords(256, 256, 256)
    kx, ky, kz = kooshball(391, 256, 100000)
    rng = np.random.default_rng(3)
    Dr, Di = _f32(rng.standard_normal(100000)), _f32(rng.standard_normal(100000))
    return Problem("3D 256^3 N=16777216, kooshball M=100000, F^H D", x, y, z, kx, ky, kz, Dr, Di, op="fhd")


def _workload_5():
    x, y, z = grid_coords(128, 128, 128)
    kx, ky, kz = stack_of_spirals(64, 4096, 64.0, 64.0)
    rng = np.random.default_rng(4)
    img = ellipsoid_image(x, y, z)
    n = x.shape[0]
    rr = img + 0.01 * rng.standard_normal(n)
    ri = 0.01 * rng.standard_normal(n)
    return Problem("3D 128^3 N=2097152, stack of spirals M=262144, F^H F rho", x, y, z, kx, ky, kz,
                   rho_r=_f32(rr), rho_i=_f32(ri), op="fhf")


WORKLOADS = {
    1: _workload_1,
    2: _workload_2,
    3: _workload_3,
    4: _workload_4,
    5: _workload_5,
}


def make_workload(i: int) -> Problem:
    """Build benchmark workload ``i`` (1..5) deterministically."""
    p = WORKLOADS[i]()
    p.meta["workload"] = i
    return p


def random_problem(N: int, M: int, kmax: float = 32.0, seed: int = 0, dims: int = 3,
                   op: str = "fhd", coords: str = "uniform") -> Problem:
    """A small random problem for parity tests.

    Voxel coordinates are uniform in [-0.5, 0.5)^dims (``coords="uniform"``)
    or the first N points of a regular grid (``coords="grid"``); k is uniform in
    [-kmax, kmax)^dims; data / image entries are standard normal.  Draw order:
    coordinates, k, real part, imaginary part.
    """
    rng = np.random.default_rng(seed)
    if coords == "grid":
        side = max(2, int(math.ceil(N ** (1.0 / dims))))
        gx, gy, gz = grid_coords(side, side, side if dims == 3 else 1)
        x, y, z = gx[:N].copy(), gy[:N].copy(), gz[:N].copy()
    else:
        c = rng.uniform(-0.5, 0.5, size=(N, dims))
        cols = [c[:, d] for d in range(dims)] + [np.zeros(N)] * (3 - dims)
        x, y, z = (_f32(v) for v in cols)
    kx, ky, kz = uniform_k(rng, M, kmax, dims)
    if op == "fhd":
        Dr, Di = _f32(rng.standard_normal(M)), _f32(rng.standard_normal(M))
        return Problem(f"random N={N} M={M}", x, y, z, kx, ky, kz, Dr, Di, op=op)
    rr, ri = _f32(rng.standard_normal(N)), _f32(rng.standard_normal(N))
    return Problem(f"random N={N} M={M} ({op})", x, y, z, kx, ky, kz, rho_r=rr, rho_i=ri, op=op)
