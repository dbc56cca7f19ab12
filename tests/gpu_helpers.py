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


def sample_indices(n: int, count: int, run: int = 32, block: int = 8192) -> np.ndarray:
    """About `count` indices spread over [0, n), chosen so that every part of
    the gather's target layout is checked.

    - An odd stride: coprime with every power of two, so the sample meets
      every position 0..run-1 of a thread's run of `run` consecutive targets
      about equally often (the recurrence's anchor at position 0 and every
      chained target after it), and every residue of a power-of-two row
      length (both row ends).
    - The first and last `run` targets of the first, a middle and the last
      target block of `block` targets (block edges, the ragged last block).
    - The last `run` targets.
    """
    if n <= count:
        return np.arange(n)
    stride = max(1, n // count)
    if stride % 2 == 0:
        stride -= 1
    idx = [np.arange(0, n, stride)[:count]]
    last_block = ((n - 1) // block) * block
    for b0 in sorted({0, ((n // block) // 2) * block, last_block}):
        idx.append(np.arange(b0, min(n, b0 + run)))
        idx.append(np.arange(max(0, b0 + block - run), min(n, b0 + block)))
    idx.append(np.arange(max(0, n - run), n))
    return np.unique(np.concatenate(idx))


def rel_l2_by_position(got, ref, idx, run: int = 32) -> dict:
    """Relative L2 error over the sampled targets at each position idx % run
    of a thread's run of consecutive targets."""
    got, ref, pos = np.asarray(got), np.asarray(ref), np.asarray(idx) % run
    return {int(q): rel_l2(got[pos == q], ref[pos == q]) for q in range(run) if np.any(pos == q)}


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


class step_records:
    """Context manager: turn the adjoint gather's step records on or off
    (fhd_test_set_step_records)."""

    def __init__(self, enable: int):
        self.enable = enable

    def __enter__(self):
        import non_cartesian_mri_gather_gb300 as fhd

        self.prev = fhd.load().fhd_test_set_step_records(self.enable)
        assert self.prev in (0, 1)
        return self

    def __exit__(self, *exc):
        import non_cartesian_mri_gather_gb300 as fhd

        fhd.load().fhd_test_set_step_records(self.prev)
        return False


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
