"""One reconstruction spread over several GPUs, one process per GPU.

The sums shard without any arithmetic outside the library's kernels:

- F^H D over voxel ranges.  Every rank holds all M samples (kx, ky, kz, D:
  20 bytes each, a few MB) and computes rho for its own contiguous range of
  voxels; the ranges are disjoint and cover the image, so nothing is
  exchanged ("Case study - iterative MRI reconstruction", section 17.3: each
  rho_n is a sum over all samples for its own voxel).
- F rho over sample ranges: every rank holds all voxels and computes D for
  its own range of samples.
- F^H F rho (section 17.3.2: the forward pass, then the adjoint pass).  With
  the image sharded by voxel ranges (as a conjugate-gradient solve keeps all
  its vectors), one application is: all-gather rho (2 N floats), the forward
  pass for this rank's sample range, all-gather F rho (2 M floats), the
  adjoint pass for this rank's voxel range.  The two exchanges are plain
  data movement (torch.distributed.all_gather); every sum runs in the
  library's gather kernels, and each rank's work is 2 N M / world pairs.

The operators default to the library's (``fhd_compute``, ``fwd_compute``),
which take CUDA tensors; ``ops`` lets a caller pass others with the same
signatures, as the CPU tests of this partitioning do with the fp64 oracle on
gloo ranks.  Every rank holds the voxel coordinates of the whole image (they
are read by the forward pass) and passes the same arrays.
"""
from __future__ import annotations


def partition(n: int, world: int, rank: int):
    """[start, stop) of rank `rank`'s contiguous share of n items: the first
    n % world ranks take one item more, so the ranges are disjoint, ordered and
    cover [0, n) exactly."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"partition: n={n} world={world} rank={rank}")
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def _default_ops():
    from . import fhd_compute, fwd_compute

    return {"fhd": fhd_compute, "fwd": fwd_compute}


def _group_info(group):
    import torch.distributed as dist

    return dist.get_world_size(group), dist.get_rank(group)


def all_gather_ranges(local, n: int, group=None):
    """Concatenate every rank's `local` (its partition() share of n items, 1-D)
    into the full length-n tensor, in rank order.  Shares are padded to the
    largest share for the collective and the padding is dropped."""
    import torch
    import torch.distributed as dist

    world, rank = _group_info(group)
    start, stop = partition(n, world, rank)
    if local.numel() != stop - start:
        raise ValueError(f"rank {rank}: {local.numel()} items, its share of {n} is {stop - start}")
    width = -(-n // world) if n else 0
    buf = torch.zeros(width, dtype=local.dtype, device=local.device)
    buf[: local.numel()] = local
    parts = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf, group=group)
    return torch.cat([parts[r][: partition(n, world, r)[1] - partition(n, world, r)[0]] for r in range(world)])


def fhd_compute_sharded(kx, ky, kz, Dr, Di, x, y, z, mode=0, group=None, ops=None):
    """This rank's share of rho = F^H D.  kx, ky, kz, Dr, Di: all M samples;
    x, y, z: all N voxels.  Returns (rho_r, rho_i) for the voxels of
    partition(N, world, rank); no exchange."""
    ops = ops or _default_ops()
    world, rank = _group_info(group)
    n0, n1 = partition(x.numel(), world, rank)
    return ops["fhd"](kx, ky, kz, Dr, Di, x[n0:n1].contiguous(), y[n0:n1].contiguous(), z[n0:n1].contiguous(),
                      mode=mode)


def fwd_compute_sharded(x, y, z, rho_r, rho_i, kx, ky, kz, mode=0, group=None, ops=None):
    """This rank's share of D = F rho.  x, y, z, rho: all N voxels; kx, ky, kz:
    all M samples.  Returns (D_r, D_i) for the samples of partition(M, world,
    rank); no exchange."""
    ops = ops or _default_ops()
    world, rank = _group_info(group)
    m0, m1 = partition(kx.numel(), world, rank)
    return ops["fwd"](x, y, z, rho_r, rho_i, kx[m0:m1].contiguous(), ky[m0:m1].contiguous(),
                      kz[m0:m1].contiguous(), mode=mode)


def fhfrho_apply_sharded(x, y, z, rho_r_local, rho_i_local, kx, ky, kz, mode=0, group=None, ops=None):
    """This rank's share of F^H F rho, with rho sharded by voxel ranges.

    x, y, z: all N voxels; rho_r_local, rho_i_local: this rank's share
    (partition(N, world, rank)); kx, ky, kz: all M samples.  Returns
    (out_r, out_i) for this rank's voxels.  Two all-gathers: rho (2 N floats)
    and F rho (2 M floats)."""
    ops = ops or _default_ops()
    N, M = x.numel(), kx.numel()
    rho_r = all_gather_ranges(rho_r_local, N, group)
    rho_i = all_gather_ranges(rho_i_local, N, group)
    Fr, Fi = fwd_compute_sharded(x, y, z, rho_r, rho_i, kx, ky, kz, mode=mode, group=group, ops=ops)
    Fr = all_gather_ranges(Fr, M, group)
    Fi = all_gather_ranges(Fi, M, group)
    return fhd_compute_sharded(kx, ky, kz, Fr, Fi, x, y, z, mode=mode, group=group, ops=ops)
