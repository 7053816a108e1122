"""The benchmark's multi-rank logic on the CPU: two gloo ranks, each with its
own timings, agree on the element-wise maximum; the barrier returns; and the
reference arm prints only on rank 0."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - rank, 3.5]
    got = bench.max_over_ranks(mine)
    total = bench.sum_over_ranks([1.0 + rank, 2.0])
    bench.barrier()
    out.put((rank, (got, total)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert res[r] == ([2.0, 10.0, 3.5], [3.0, 4.0])


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]


def test_reference_arm_quiet_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120)
    assert proc.returncode == 0
    assert proc.stdout.strip() == ""


def test_clock_samples_that_invalidate_a_run():
    import bench

    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"]))  # kept and noted
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[r]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1200.0))  # stuck low with no reason: a clock lock
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1200.0, reasons=["sw_power_cap"]))
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]})


def test_shard_map_slab_workloads_cover_the_grid():
    """--shard-map: the ranks' slab workloads hold all atoms and together
    exactly the full grid's planes, cutoff slabs in whole 8-plane bricks."""
    import workloads

    sys.path.insert(0, ROOT)
    import bench

    w = workloads.make("cutoff_uniform")
    for world in (1, 2, 3, 4):
        slabs = [bench.slab_workload(w, r, world, 8) for r in range(world)]
        assert sum(s.shape[2] for s in slabs) == w.shape[2]
        for s in slabs:
            assert s.shape[:2] == w.shape[:2] and s.atoms is w.atoms
        zs = [round((s.origin[2] - w.origin[2]) / w.h) for s in slabs]
        assert zs == sorted(zs) and all(z % 8 == 0 for z in zs)
