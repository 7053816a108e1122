"""Z-slab sharding on the CPU: the slab arithmetic of cp_slab, and the gather
of slabs over gloo ranks (2 and 3 processes) into the full map.  The slab
maps here come from the oracle on each rank's slab grid, so the assembled
map must equal the oracle's map of the whole grid bit for bit: the slab
grids hold exactly the full grid's points, and every point's sum is the
same sequence of fp64 operations."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _slab(*a):
    from direct_coulomb_summation_gb300 import shard

    return shard.slab(*a)


@pytest.mark.parametrize("nz", [1, 7, 8, 9, 64, 200, 401])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8, 13])
@pytest.mark.parametrize("align", [1, 8])
def test_slabs_cover_the_grid_in_rank_order(nz, world, align):
    slabs = [_slab(nz, world, r, align, 0.0, 0.5) for r in range(world)]
    z = 0
    units = -(-nz // align)
    for r, (z0, n, oz) in enumerate(slabs):
        assert z0 == z and n >= 0
        assert z0 % align == 0
        # whole units except where nz cuts the last one short
        assert n % align == 0 or z0 + n == nz
        # units shared as evenly as integer division allows
        u = -(-n // align) if n else 0
        assert u in (units // world, units // world + 1)
        assert oz == np.float32(z0 * 0.5)
        z += n
    assert z == nz


@pytest.mark.parametrize("oz,h,z0_world_rank", [(1.25, 0.37, (5, 8, 7)), (-3.0, 0.5, (100, 3, 2)),
                                                 (5000.0, 0.37, (64, 2, 1))])
def test_slab_origin_is_the_full_grids_plane(oz, h, z0_world_rank):
    """The slab origin is fp32(z0*h + origin_z) rounded once, the coordinate
    the kernels give plane z0 of the full grid."""
    nz, world, rank = z0_world_rank
    z0, n, ozs = _slab(nz, world, rank, 1, oz, h)
    exact = float(np.float32(oz)) + z0 * float(np.float32(h))  # exact in fp64 for these values
    assert ozs == float(np.float32(exact))


@pytest.mark.parametrize("args", [(0, 1, 0, 1), (8, 0, 0, 1), (8, 2, 2, 1), (8, 2, -1, 1), (8, 2, 0, 0)])
def test_slab_rejects_bad_arguments(args):
    import direct_coulomb_summation_gb300 as cp

    with pytest.raises(cp.CpError):
        _slab(*args, 0.0, 0.5)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, kind, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    import workloads
    from direct_coulomb_summation_gb300 import shard

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w = workloads.random_case(71, 300, (9, 7, 19), h=0.5, origin=(-1.0, 0.5, 2.0), margin=3.0)
        align = shard.BRICK_PLANES if kind == "cutoff" else 1
        z0, sshape, sorigin = shard.slab_grid(w.shape, w.origin, w.h, rank, world, align)
        V = None
        if sshape[2] > 0:
            if kind == "direct":
                v, _ = oracle.direct(w.atoms, sshape, sorigin, w.h)
            else:
                v, _ = oracle.cutoff_brute(w.atoms, sshape, sorigin, w.h, 3.0)
            V = torch.from_numpy(np.asarray(v, dtype=np.float64).reshape(sshape[2], sshape[1], sshape[0]))
            V = V.float()
        full = shard.gather_slabs(V, w.shape, align, dst=0)
        if rank == 0:
            if kind == "direct":
                ref, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h)
            else:
                ref, _ = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, 3.0)
            ref = np.asarray(ref, dtype=np.float64).astype(np.float32).reshape(w.shape[2], w.shape[1], w.shape[0])
            out.put((rank, bool(np.array_equal(full.numpy(), ref)), tuple(full.shape)))
        else:
            out.put((rank, full is None, None))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("kind", ["direct", "cutoff"])
def test_gather_assembles_the_full_map(world, kind):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, kind, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, ok, shape = q.get(timeout=180)
        res[r] = (ok, shape)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(ok for ok, _ in res.values()), res
    assert res[0][1] == (19, 7, 9)
