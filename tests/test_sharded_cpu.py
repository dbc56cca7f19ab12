"""The multi-GPU partitioning (non_cartesian_mri_gather_gb300.sharded) on the
CPU: partition() covers every index once, and on two and three gloo ranks the
sharded F^H D, F rho and F^H F rho, run with the fp64 oracle as the local
operator, concatenate to exactly the oracle's result on the whole problem
(each output of a gather sum depends only on its own voxel or sample, so a
share computes bit for bit what the whole computes there).  Sizes are not
divisible by the rank count."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from non_cartesian_mri_gather_gb300.sharded import partition  # noqa: E402

N, M = 1001, 333


@pytest.mark.parametrize("n", [0, 1, 5, 7, 1000, 2 ** 24 + 3])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_partition_covers_once(n, world):
    ranges = [partition(n, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0 and a0 <= a1
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_partition_rejects_bad_arguments():
    for args in ((5, 0, 0), (5, 2, 2), (5, 2, -1), (-1, 2, 0)):
        with pytest.raises(ValueError):
            partition(*args)


def _problem():
    rng = np.random.default_rng(70)
    x, y, z = (rng.uniform(-0.5, 0.5, N).astype(np.float32) for _ in range(3))
    kx, ky, kz = (rng.uniform(-16, 16, M).astype(np.float32) for _ in range(3))
    D = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    rho = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    return x, y, z, kx, ky, kz, D, rho


def _oracle_ops():
    """The fp64 oracle behind the library operators' signatures (CPU tensors)."""
    import torch

    import oracle

    def fhd(kx, ky, kz, Dr, Di, x, y, z, mode=0):
        r = oracle.adjoint(kx.numpy(), ky.numpy(), kz.numpy(), Dr.numpy() + 1j * Di.numpy(), x.numpy(), y.numpy(),
                           z.numpy())
        return torch.from_numpy(r.real.copy()), torch.from_numpy(r.imag.copy())

    def fwd(x, y, z, rr, ri, kx, ky, kz, mode=0):
        r = oracle.forward(x.numpy(), y.numpy(), z.numpy(), rr.numpy() + 1j * ri.numpy(), kx.numpy(), ky.numpy(),
                           kz.numpy())
        return torch.from_numpy(r.real.copy()), torch.from_numpy(r.imag.copy())

    return {"fhd": fhd, "fwd": fwd}


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from non_cartesian_mri_gather_gb300 import sharded

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, y, z, kx, ky, kz, D, rho = (torch.from_numpy(np.ascontiguousarray(a)) for a in _problem())
        ops = _oracle_ops()
        a = sharded.fhd_compute_sharded(kx, ky, kz, D.real.contiguous(), D.imag.contiguous(), x, y, z, ops=ops)
        b = sharded.fwd_compute_sharded(x, y, z, rho.real.contiguous(), rho.imag.contiguous(), kx, ky, kz, ops=ops)
        n0, n1 = sharded.partition(N, world, rank)
        c = sharded.fhfrho_apply_sharded(x, y, z, rho.real[n0:n1].contiguous(), rho.imag[n0:n1].contiguous(), kx, ky,
                                         kz, ops=ops)
        for name, (re, im) in (("fhd", a), ("fwd", b), ("fhf", c)):
            np.save(os.path.join(out, f"{name}_{rank}.npy"), re.numpy() + 1j * im.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_operators_gloo(tmp_path, world):
    import torch.multiprocessing as mp

    import oracle

    oracle.get()  # build the oracle once, before the ranks start
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn", join=True)
    x, y, z, kx, ky, kz, D, rho = _problem()
    got = {name: np.concatenate([np.load(tmp_path / f"{name}_{r}.npy") for r in range(world)])
           for name in ("fhd", "fwd", "fhf")}
    assert got["fhd"].shape == (N,) and got["fwd"].shape == (M,) and got["fhf"].shape == (N,)
    assert np.array_equal(got["fhd"], oracle.adjoint(kx, ky, kz, D, x, y, z))
    assert np.array_equal(got["fwd"], oracle.forward(x, y, z, rho, kx, ky, kz))
    assert np.array_equal(got["fhf"], oracle.normal(x, y, z, rho, kx, ky, kz))
