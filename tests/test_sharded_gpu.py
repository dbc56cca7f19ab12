"""The multi-GPU partitioning (non_cartesian_mri_gather_gb300.sharded) with the
library's own operators on the GPU: a one-rank NCCL process group runs the
sharded F^H D, F rho and F^H F rho (its two all-gathers included), and each
result is bit-identical to the unsharded library call, which with one rank
computes the same gathers.  The partitioning over several ranks is checked
on CPU ranks (test_sharded_cpu.py); every run here has one GPU."""
import socket

import numpy as np
import pytest

from inputs import random_problem
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def group():
    import torch
    import torch.distributed as dist

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from non_cartesian_mri_gather_gb300 import build, load

    build.build()
    load()
    torch.cuda.set_device(0)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("mode", [0, 1])
def test_sharded_operators_one_rank(group, mode):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd
    from non_cartesian_mri_gather_gb300 import sharded

    p = random_problem(20000, 3000, kmax=24.0, seed=80, op="fhf", coords="grid")
    t = {k: dev(getattr(p, k)) for k in ("x", "y", "z", "kx", "ky", "kz", "rho_r", "rho_i")}
    Dr, Di = t["rho_r"][: p.M].contiguous(), t["rho_i"][: p.M].contiguous()
    a = sharded.fhd_compute_sharded(t["kx"], t["ky"], t["kz"], Dr, Di, t["x"], t["y"], t["z"], mode=mode)
    a0 = fhd.fhd_compute(t["kx"], t["ky"], t["kz"], Dr, Di, t["x"], t["y"], t["z"], mode=mode)
    b = sharded.fwd_compute_sharded(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"],
                                    mode=mode)
    b0 = fhd.fwd_compute(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"], mode=mode)
    c = sharded.fhfrho_apply_sharded(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"],
                                     mode=mode)
    c0 = fhd.fhfrho_apply(t["x"], t["y"], t["z"], t["rho_r"], t["rho_i"], t["kx"], t["ky"], t["kz"], mode=mode)
    torch.cuda.synchronize()
    for got, want in ((a, a0), (b, b0), (c, c0)):
        assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])
        assert bool(torch.isfinite(got[0]).all()) and bool(torch.isfinite(got[1]).all())
    assert np.isfinite(c[0].sum().item())
