"""Z-slab sharding on the GPU: two processes share the one GPU, each computes
its slab with the library's kernels and the slabs are gathered over gloo
(host copies).  The two processes' kernels are independent launches that
never wait on each other.

  * direct map, patch shape and cluster split forced equal to the single
    call's: the assembled map equals the single-call map bit for bit;
  * cutoff map (brick-aligned slabs, capacity 0 and 16): within the oracle's
    bound, checked on sampled points of the assembled map."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, kind, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import direct_coulomb_summation_gb300 as cp
    import workloads
    from direct_coulomb_summation_gb300 import shard

    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        if kind == "direct":
            w = workloads.make("direct_3d")
            v, sp = cp.direct_plan(w.n_atoms, w.shape)
            full = shard.direct_sharded(torch.from_numpy(w.atoms).cuda(), w.shape, w.origin, w.h, variant=v,
                                        split=sp)
        else:
            w = workloads.make("cutoff_uniform")
            K = int(kind.split("_")[1])
            full = shard.cutoff_sharded(torch.from_numpy(w.atoms).cuda(), w.shape, w.origin, w.h, w.cutoff,
                                        w.bin_size, K)
        torch.cuda.synchronize()
        status = cp.device_status()
        if rank == 0:
            np.save(os.path.join(out_dir, f"{kind}.npy"), full.cpu().numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()
    if status != 0:
        raise RuntimeError(f"device status {status:#x}")


def _run_ranks(kind, tmp_path, world=2):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, kind, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    return np.load(os.path.join(tmp_path, f"{kind}.npy"))


def test_direct_sharded_equals_single_call(tmp_path):
    import direct_coulomb_summation_gb300 as cp
    import workloads

    got = _run_ranks("direct", tmp_path)
    w = workloads.make("direct_3d")
    v, sp = cp.direct_plan(w.n_atoms, w.shape)
    ref = cp.direct(torch.from_numpy(w.atoms).cuda(), w.shape, w.origin, w.h, variant=v, split=sp)
    torch.cuda.synchronize()
    assert got.shape == tuple(ref.shape)
    assert np.array_equal(got, ref.cpu().numpy())


@pytest.mark.parametrize("K", [0, 16])
def test_cutoff_sharded_within_oracle_bound(tmp_path, K):
    import oracle
    import workloads
    from gpu_util import assert_within_bound, flat_index

    got = _run_ranks(f"cutoff_{K}", tmp_path)
    w = workloads.make("cutoff_uniform")
    assert got.shape == (w.shape[2], w.shape[1], w.shape[0])
    # sampled points plus every point of the two planes either side of the slab boundary
    nx, ny, nz = w.shape
    ij = np.stack(np.meshgrid(np.arange(nx), np.arange(ny), indexing="xy"), -1).reshape(-1, 2)
    edge = np.concatenate([np.column_stack([ij, np.full(len(ij), z)]) for z in (95, 96)])
    pts = np.concatenate([workloads.sample_points(w.shape, 2048, seed=4200), edge])
    ref, bound = oracle.cutoff_binned(w.atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, points=pts)
    assert_within_bound(got.reshape(-1)[flat_index(w.shape, pts)], ref, bound, f"sharded cutoff K={K}")
