"""Z-slab sharding of a potential map over the ranks of a torch.distributed
group (one process per GPU).

Grid points are independent: each is written only by the thread that owns
it (PMPP ch.18 notes, section 18.2, the gather formulation), so a map splits
into slabs of whole z-planes that separate GPUs compute without exchanging
anything.  The direct sum needs every atom on every rank; the cutoff sum
needs only the atoms within c of a rank's slab, and the bin rule of the
slab's own grid keeps exactly those (section 18.5: bins bound each point's
atoms to its neighbourhood), so every rank is handed all atoms and drops the
rest while binning.  The slabs are then gathered to one owner rank.

The slab arithmetic is the library's ``cp_slab`` (host-only C ABI); every
slab is computed by the ordinary ``cp_direct`` / ``cp_cutoff`` calls on the
slab's sub-grid, and the gather is a torch.distributed collective of plain
device (NCCL) or host (gloo) tensors.

    from direct_coulomb_summation_gb300 import shard
    V = shard.direct_sharded(atoms, (nx, ny, nz), origin, h)      # full map on rank 0
    V = shard.cutoff_sharded(atoms, (nx, ny, nz), origin, h, 12.0, 4.0)
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch
import torch.distributed as dist

from . import _check, _lib, cutoff, direct

__all__ = ["slab", "slab_grid", "direct_slab", "cutoff_slab", "gather_slabs", "direct_sharded",
           "cutoff_sharded", "BRICK_PLANES"]

# planes per slab unit for the cutoff map: its bricks are 8x8x8 points
BRICK_PLANES = 8


def slab(nz: int, world: int, rank: int, align: int = 1, origin_z: float = 0.0, h: float = 1.0):
    """(z0, nz_slab, origin_z_slab) of rank `rank` of `world` (``cp_slab``)."""
    z0, n, oz = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_float(0.0)
    rc = _lib.load().cp_slab(int(nz), int(world), int(rank), int(align), float(np.float32(origin_z)),
                             float(np.float32(h)), ctypes.byref(z0), ctypes.byref(n), ctypes.byref(oz))
    _check(rc, "cp_slab")
    return int(z0.value), int(n.value), float(oz.value)


def slab_grid(shape, origin, h, rank: int, world: int, align: int = 1):
    """(z0, slab shape, slab origin) of a rank's slab of the grid."""
    nx, ny, nz = (int(s) for s in shape)
    z0, n, oz = slab(nz, world, rank, align, origin[2], h)
    return z0, (nx, ny, n), (float(np.float32(origin[0])), float(np.float32(origin[1])), oz)


def _rank_world(group, rank, world):
    if rank is None or world is None:
        if not (dist.is_available() and dist.is_initialized()):
            return 0, 1
        return dist.get_rank(group), dist.get_world_size(group)
    return int(rank), int(world)


def direct_slab(atoms, shape, origin, h, rank: Optional[int] = None, world: Optional[int] = None, align: int = 1,
                group=None, out=None, stream=None, variant: int = -1, split: int = 0):
    """This rank's slab of the direct map as (z0, V_slab), V_slab of shape
    (nz_slab, ny, nx) on the current GPU (None for an empty slab).  Every
    rank passes all atoms."""
    rank, world = _rank_world(group, rank, world)
    z0, sshape, sorigin = slab_grid(shape, origin, h, rank, world, align)
    if sshape[2] == 0:
        return z0, None
    return z0, direct(atoms, sshape, sorigin, h, out=out, stream=stream, variant=variant, split=split)


def cutoff_slab(atoms, shape, origin, h, cutoff_radius, bin_size, capacity: int = 0, rank: Optional[int] = None,
                world: Optional[int] = None, align: int = BRICK_PLANES, group=None, workspace=None, out=None,
                stream=None):
    """This rank's slab of the cutoff map as (z0, V_slab); every rank passes
    all atoms, and binning on the slab's grid drops those farther than the
    cutoff from the slab (the atom halo needs no exchange)."""
    rank, world = _rank_world(group, rank, world)
    z0, sshape, sorigin = slab_grid(shape, origin, h, rank, world, align)
    if sshape[2] == 0:
        return z0, None
    return z0, cutoff(atoms, sshape, sorigin, h, cutoff_radius, bin_size, capacity, workspace=workspace, out=out,
                      stream=stream)


def gather_slabs(V_slab, shape, align: int = 1, group=None, dst: int = 0, rank: Optional[int] = None,
                 world: Optional[int] = None):
    """Gathers every rank's slab (z0 order = rank order) into the full map
    (nz, ny, nx) on rank `dst`; returns None on the other ranks.  Slabs are
    padded to the largest slab's planes for the collective.  With the gloo
    backend the collective runs on host copies; the full map is returned on
    the device V_slab came from."""
    rank, world = _rank_world(group, rank, world)
    nx, ny, nz = (int(s) for s in shape)
    sizes = [slab(nz, world, r, align)[1] for r in range(world)]
    if world == 1:
        return V_slab if V_slab is not None else torch.zeros((0, ny, nx), dtype=torch.float32)
    backend = dist.get_backend(group)
    home = V_slab.device if V_slab is not None else torch.device("cpu")
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    pad = torch.zeros((max(sizes), ny, nx), dtype=torch.float32, device=dev)
    if V_slab is not None and sizes[rank] > 0:
        pad[: sizes[rank]].copy_(V_slab.reshape(sizes[rank], ny, nx))
    parts = [torch.empty_like(pad) for _ in range(world)] if rank == dst else None
    dist.gather(pad, parts, dst=dst, group=group)
    if rank != dst:
        return None
    full = torch.cat([p[:n] for p, n in zip(parts, sizes)], dim=0)
    return full.to(home) if home.type == "cuda" else full


def direct_sharded(atoms, shape, origin, h, group=None, dst: int = 0, variant: int = -1, split: int = 0):
    """The direct map computed as z-slabs on every rank of `group` and
    gathered to rank `dst` (None elsewhere)."""
    _, V = direct_slab(atoms, shape, origin, h, group=group, variant=variant, split=split)
    return gather_slabs(V, shape, 1, group=group, dst=dst)


def cutoff_sharded(atoms, shape, origin, h, cutoff_radius, bin_size, capacity: int = 0, group=None, dst: int = 0):
    """The cutoff map computed as brick-aligned z-slabs on every rank of
    `group` and gathered to rank `dst` (None elsewhere)."""
    _, V = cutoff_slab(atoms, shape, origin, h, cutoff_radius, bin_size, capacity, group=group)
    return gather_slabs(V, shape, BRICK_PLANES, group=group, dst=dst)
