"""Helpers for the GPU tests: device copies, error metrics, sampled oracle checks."""
from __future__ import annotations

import numpy as np

# Tolerances on the relative L2 error against the fp64 oracle.
TOL_ACCURATE = 1e-5
TOL_FAST = 1e-3
PSNR_FAST_DB = 60.0


def rel_l2(got, ref) -> float:
    got, ref = np.asarray(got), np.asarray(ref)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def psnr_db(got, ref) -> float:
    """20 log10(max|ref| / RMSE) over the complex values."""
    got, ref = np.asarray(got), np.asarray(ref)
    rmse = np.sqrt(np.mean(np.abs(got - ref) ** 2))
    return float(20 * np.log10(np.max(np.abs(ref)) / max(rmse, 1e-300)))


def dev(a, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_complex(re, im) -> np.ndarray:
    return re.detach().cpu().numpy().astype(np.float64) + 1j * im.detach().cpu().numpy().astype(np.float64)


def sample_indices(n: int, count: int, seed: int = 0) -> np.ndarray:
    """A fixed spread of indices: evenly strided plus the first and last few."""
    if n <= count:
        return np.arange(n)
    stride = max(1, n // count)
    idx = np.arange(0, n, stride)[:count]
    tail = np.arange(max(0, n - 5), n)
    return np.unique(np.concatenate([idx, np.arange(5), tail]))


def gpu_fhd(p, mode, ws=None):
    import non_cartesian_mri_gather_gb300 as fhd
    import torch

    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "Dr", "Di")}
    rr, ri = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], t["Dr"], t["Di"], t["x"], t["y"], t["z"], mode=mode,
                             workspace=ws)
    torch.cuda.synchronize()
    return host_complex(rr, ri)


def gpu_fwd(p, mode, rho=None):
    import non_cartesian_mri_gather_gb300 as fhd
    import torch

    rr = p.rho_r if rho is None else rho.real.astype(np.float32)
    ri = p.rho_i if rho is None else rho.imag.astype(np.float32)
    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz")}
    Dr, Di = fhd.fwd_compute(t["x"], t["y"], t["z"], dev(rr), dev(ri), t["kx"], t["ky"], t["kz"], mode=mode)
    torch.cuda.synchronize()
    return host_complex(Dr, Di)


def gpu_fhf(p, mode):
    import non_cartesian_mri_gather_gb300 as fhd
    import torch

    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "rho_r", "rho_i")}
    o_r, o_i = fhd.fhfrho_apply(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"], mode=mode)
    torch.cuda.synchronize()
    return host_complex(o_r, o_i)


PATH_AUTO, PATH_PERSISTENT, PATH_SPLIT = 0, 1, 2


class gather_path:
    """Context manager: force the library's gather path (fhd_test_set_path)."""

    def __init__(self, path: int):
        self.path = path

    def __enter__(self):
        import non_cartesian_mri_gather_gb300 as fhd

        self.prev = fhd.load().fhd_test_set_path(self.path)
        assert self.prev in (0, 1, 2)
        return self

    def __exit__(self, *exc):
        import non_cartesian_mri_gather_gb300 as fhd

        fhd.load().fhd_test_set_path(self.prev)
        return False
