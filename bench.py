#!/usr/bin/env python
"""Benchmark of the potential-map hot path on GB300.

One step = the whole hot path over one batch of synthetic input, on the two
largest single-GPU workloads:
  * direct map (D1-D5): 200^3 grid (8,000,000 points) at h = 0.5 A, 100,000
    off-lattice atoms from 200 Gaussian clusters, charges in
    {-1, -0.5, 0.5, 1}  ->  pair evaluations/s (the headline ``value``);
  * cutoff map (C1-C6): 400^3 grid (64,000,000 points) at h = 0.5 A,
    800,000 atoms (70 % uniform, 30 % in 500 Gaussian clusters), c = 12 A,
    4 A bins, capacity 0 (each bin a contiguous bin-sorted run, no fixed
    slots): on-device binning then the brick map  ->  grid points/s and
    useful pairs/s.
After the timed steps every other workload is timed on its own with the
pwwt.cn article's protocol (3 warm-ups, 10 timed runs): the 100x100 plane
and the 128x128x64 direct maps, the 200^3 / 100k-atom cutoff map at
capacity 0, and both cutoff maps with the lecture's fixed-capacity bins
plus overflow list (capacity 8 and 16), each with its roofline fraction.
Inputs are resident in HBM; L2 is flushed (a 256 MiB write) before every
timed launch; each launch is timed with CUDA events on its stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own copy
of the step (weak scaling, no collective on the data path); timings are the
max over ranks.  ``--impl reference`` times the fp64 CPU oracle on the host
cores instead, on bounded samples of the same direct workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "pair evals/s (direct Coulomb) and grid points/s at 12 Å cutoff, % of roofline"
DIRECT_WL = "direct_protein"   # 200^3, 100k clustered atoms
CUTOFF_WL = "cutoff_large"     # 400^3, 800k atoms, c = 12 A
CAPACITY_DEFAULT = 0
FLUSH_BYTES = 256 << 20
# the other workloads, timed one by one after the steps
SECONDARY_DIRECT = ["direct_plane", "direct_3d"]
SECONDARY_CUTOFF = [("cutoff_uniform", 0), ("cutoff_uniform", 8), ("cutoff_uniform", 16),
                    ("cutoff_large", 8), ("cutoff_large", 16)]
CONFIG_NUMBER = {"direct_plane": 1, "direct_3d": 2, "direct_protein": 3, "cutoff_uniform": 4, "cutoff_large": 5}


def env_rank():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def config_dict(wd, wc, capacity, shards=0):
    return {
        "workload": f"direct {wd.shape[0]}x{wd.shape[1]}x{wd.shape[2]} grid, {wd.n_atoms} clustered atoms, "
        f"h={wd.h} A (config {CONFIG_NUMBER.get(wd.meta.get('key', ''), '?')}); "
        f"cutoff {wc.shape[0]}x{wc.shape[1]}x{wc.shape[2]} grid, {wc.n_atoms} atoms, c={wc.cutoff} A, "
        f"{wc.bin_size} A bins, bin capacity {capacity} "
        f"({'contiguous bin-sorted runs, no fixed slots' if capacity == 0 else 'fixed slots + overflow list'}) "
        f"(config {CONFIG_NUMBER.get(wc.meta.get('key', ''), '?')})",
        "direct": {"grid": list(wd.shape), "atoms": wd.n_atoms, "h": wd.h, "pairs": wd.n_pairs,
                   "description": wd.description},
        "cutoff": {"grid": list(wc.shape), "atoms": wc.n_atoms, "h": wc.h, "cutoff": wc.cutoff,
                   "bin_size": wc.bin_size, "capacity": capacity, "brick": [8, 8, 8],
                   "description": wc.description},
        "l2": "flushed before every timed launch (256 MiB write)",
        "parallelism": (f"one map shared by {shards} ranks as z-slabs, each rank all atoms (strong scaling)"
                        if shards else "one independent copy per rank (weak scaling)"),
    }


def slab_workload(w, rank, world, align):
    """The rank's z-slab of workload `w` (same atoms, the slab's grid)."""
    import dataclasses

    from direct_coulomb_summation_gb300 import shard

    _, shape, origin = shard.slab_grid(w.shape, w.origin, w.h, rank, world, align)
    return dataclasses.replace(w, shape=shape, origin=origin, meta=dict(w.meta))


def make_workload(name):
    import workloads

    w = workloads.make(name)
    w.meta["key"] = name
    return w


# ---------------------------------------------------------------------------
# multi-rank helpers (also exercised by tests/test_bench_ranks.py with gloo)

def max_over_ranks(values, device=None):
    """Elementwise max of a list of floats over all ranks (identity at world size 1)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def sum_over_ranks(values, device=None):
    """Elementwise sum of a list of numbers over all ranks (identity at world size 1)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.cpu().tolist()


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampled during the timed region

CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        self.t_begin = None
        self.t_end = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t_begin = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if self.t_begin is not None and not (self.t_begin <= ts <= (self.t_end or ts)):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
        }


REJECTING_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def clocks_rejected(clocks) -> bool:
    """A timed region whose clock samples show a hardware or thermal slowdown,
    or an SM clock well below its maximum with no reason (a leftover clock
    lock), is not a valid measurement."""
    if REJECTING_REASONS & set(clocks.get("reasons") or []):
        return True
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.85 * smax and not clocks.get("reasons"))


def gpu_id_for(torch, device) -> str:
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        if uuid:
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[device.index]
    return str(device.index)


# ---------------------------------------------------------------------------
# CPU baselines (the fp64 oracle, as it stands)

def oracle_direct_rate(wd, target_s: float, threads: int, seed: int = 99):
    """Times the oracle's direct sum on a sample of grid points sized for
    about target_s seconds; returns (pairs/s, n_points, seconds)."""
    import oracle
    import workloads

    n_pts = 64
    while True:
        pts = workloads.sample_points(wd.shape, n_pts, seed=seed)
        t0 = time.perf_counter()
        oracle.direct(wd.atoms, wd.shape, wd.origin, wd.h, points=pts, threads=threads, with_bound=False)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or n_pts >= wd.n_points:
            return n_pts * wd.n_atoms / dt, n_pts, dt
        n_pts = min(wd.n_points, int(n_pts * max(2.0, min(16.0, target_s / max(dt, 1e-3)))))


def oracle_cutoff_rate(wc, target_s: float, threads: int, seed: int = 98):
    import oracle
    import workloads

    n_pts = 64
    while True:
        pts = workloads.sample_points(wc.shape, n_pts, seed=seed)
        t0 = time.perf_counter()
        oracle.cutoff_binned(wc.atoms, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, points=pts,
                             threads=threads, with_bound=False)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or n_pts >= wc.n_points:
            return n_pts / dt, n_pts, dt
        n_pts = min(wc.n_points, int(n_pts * max(2.0, min(16.0, target_s / max(dt, 1e-3)))))


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores

def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return 0
    import oracle  # noqa: F401  (built on first use)
    import workloads

    wd = make_workload(DIRECT_WL)
    wc = make_workload(CUTOFF_WL)
    threads = host_threads()
    # size one step for about 1.5 s so that warm-up + steps end within minutes
    _, n_pts, _ = oracle_direct_rate(wd, 1.5, threads)
    pts = workloads.sample_points(wd.shape, n_pts, seed=99)
    import oracle as orc

    times = []
    for step in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        orc.direct(wd.atoms, wd.shape, wd.origin, wd.h, points=pts, threads=threads, with_bound=False)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
    t = sum(times)
    value = n_pts * wd.n_atoms * len(times) / t
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "pair evals/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * t / len(times),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": config_dict(wd, wc, args.capacity),
        "cpu_baseline": {"value": value, "unit": "pair evals/s", "cores": threads, "kind": "oracle",
                         "sample": f"direct sum at {n_pts} seeded grid points of the {wd.shape} grid x "
                                   f"{wd.n_atoms} atoms per step"},
        "e2e": {"value": value, "unit": "pair evals/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm

def traffic_from_profile(kernel: str, source: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if the kernel's source is unchanged since it was captured (else
    None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
        with open(os.path.join(ROOT, source), "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()
    except (OSError, ValueError, AttributeError):
        return None
    if not rec or rec.get("source_sha1") != sha:
        return None
    return (rec.get("per_workload") or {}).get(workload)


def e2e_times(cp, wd, wc, Vd, Vc, ws, host_atoms_d, host_out_d, host_atoms_c, host_out_c, n, capacity,
              do_direct=True, do_cutoff=True):
    """Seconds per call of the public API with host buffers: pinned atoms in,
    host V out, copies and synchronisation included (one untimed call first)."""
    t_d = t_c = float("nan")
    if do_direct:
        cp.direct(host_atoms_d, wd.shape, wd.origin, wd.h, out=Vd, host_out=host_out_d)
        t0 = time.perf_counter()
        for _ in range(n):
            cp.direct(host_atoms_d, wd.shape, wd.origin, wd.h, out=Vd, host_out=host_out_d)
        t_d = (time.perf_counter() - t0) / n
    if do_cutoff:
        cp.cutoff(host_atoms_c, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, capacity, workspace=ws, out=Vc,
                  host_out=host_out_c)
        t0 = time.perf_counter()
        for _ in range(n):
            cp.cutoff(host_atoms_c, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, capacity, workspace=ws,
                      out=Vc, host_out=host_out_c)
        t_c = (time.perf_counter() - t0) / n
    return t_d, t_c


class Roofline:
    """Per-SM bounds behind every roofline fraction in the line, from the
    pipe rates measured on this GPU in the same run and the SM clock sampled
    during the timed steps."""

    def __init__(self, r_mufu, r_ffma, n_sm, f_mhz, clock_basis):
        self.r_mufu, self.r_ffma, self.n_sm, self.f_mhz, self.clock_basis = r_mufu, r_ffma, n_sm, f_mhz, clock_basis
        self.sm_clk = n_sm * f_mhz * 1e6  # SM clock cycles per second, one GPU
        # direct: per pair at least 1 SFU rsqrt, 3 FP32 ops (dx, r^2,
        # accumulate) and 4 issue slots: pairs/clk/SM = min(R_sfu, R_fp32/3, 128/4)
        self.direct_sfu = min(r_mufu, r_ffma / 3.0, 32.0)
        # the same pair with its rsqrt split between the SFU and the FMA pipe
        # (estimate + two Newton steps: 6 FP32 ops): the best share f solves
        # (1 - f)/R_sfu = (3 + 6f)/R_fp32
        self.f_split = (r_ffma - 3.0 * r_mufu) / (r_ffma + 6.0 * r_mufu)
        self.direct_split = r_mufu / (1.0 - self.f_split)
        # cutoff: a useful pair needs 1 SFU rsqrt and about 11 FP32 ops (dx,
        # dy, dz, three for r^2, compare, two for g, subtract, accumulate):
        # useful pairs/clk/SM = min(R_sfu, R_fp32/11)
        self.useful = min(r_mufu, r_ffma / 11.0)
        # tighter: dy, dz and the row sums amortised over a thread's points,
        # 8 issue slots and one SFU op per useful pair: min(R_sfu, 128/8)
        self.useful_tight = min(r_mufu, 16.0)

    def direct(self, pairs_per_s, world=1):
        peak = self.direct_split * self.sm_clk * world
        peak_sfu = self.direct_sfu * self.sm_clk * world
        return {"achieved": pairs_per_s, "peak": peak, "frac": pairs_per_s / peak,
                "peak_sfu_only": peak_sfu, "frac_sfu_only": pairs_per_s / peak_sfu}

    def cutoff(self, useful_per_s, world=1):
        peak = self.useful * self.sm_clk * world
        tight = self.useful_tight * self.sm_clk * world
        return {"achieved": useful_per_s, "peak": peak, "unit": "useful pair evals/s",
                "frac": useful_per_s / peak,
                "time_vs_useful_pair_roofline": peak / useful_per_s if useful_per_s > 0 else None,
                "time_vs_tight_bound": tight / useful_per_s if useful_per_s > 0 else None}


def bin_bytes_of(L, n_atoms, capacity):
    """HBM bytes binning must move at least: atoms in, bin-sorted atoms and
    indices out, counts and starts, fixed-capacity slots out."""
    return 16 * n_atoms * 2 + 4 * n_atoms + 8 * int(L.nbins) + 16 * capacity * int(L.nbins)


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = env_rank()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (use --impl reference for the CPU oracle)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", rank=rank, world_size=world, device_id=device)

    import direct_coulomb_summation_gb300 as cp

    lib = cp.library()
    props = torch.cuda.get_device_properties(device)
    n_sm = props.multi_processor_count

    wd_full = make_workload(args.direct_workload)
    wc_full = make_workload(args.cutoff_workload)
    wd, wc = wd_full, wc_full
    if args.shard_map:
        # strong scaling: the ranks share one map, each computing a z-slab
        wd = slab_workload(wd_full, rank, world, 1)
        wc = slab_workload(wc_full, rank, world, 8)
        if wd.shape[2] == 0 or wc.shape[2] == 0:
            raise RuntimeError("--shard-map: more ranks than slabs")
    # how many full workloads one timed step covers, over all ranks
    job = 1 if args.shard_map else world
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    ad = torch.from_numpy(wd.atoms).to(device)
    Vd = torch.empty((wd.shape[2], wd.shape[1], wd.shape[0]), dtype=torch.float32, device=device)
    ac = torch.from_numpy(wc.atoms).to(device)
    Vc = torch.empty((wc.shape[2], wc.shape[1], wc.shape[0]), dtype=torch.float32, device=device)
    ws_bytes = cp.cutoff_workspace_bytes(wc.n_atoms, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, args.capacity)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    gd = cp._grid(wd.shape, wd.origin, wd.h)
    gc = cp._grid(wc.shape, wc.origin, wc.h)
    cut = [float(np.float32(wc.cutoff)), float(np.float32(wc.bin_size)), args.capacity]

    def call(rc, where):
        if rc != 0:
            raise cp.CpError(rc, where)

    def run_direct():
        call(lib.cp_direct(ad.data_ptr(), wd.n_atoms, *gd, Vd.data_ptr(), sh), "cp_direct")

    def run_bin():
        call(lib.cp_bin_atoms(ac.data_ptr(), wc.n_atoms, *gc, *cut, ws.data_ptr(), ws_bytes, sh), "cp_bin_atoms")

    def run_map():
        call(lib.cp_cutoff_map(ac.data_ptr(), wc.n_atoms, *gc, *cut, ws.data_ptr(), ws_bytes, Vc.data_ptr(), sh),
             "cp_cutoff_map")

    # roofline denominators: per-SM pipe rates measured on this GPU
    r_mufu, _ = cp.probe_pipe_rate("mufu_rsqrt", 32, 4096)
    r_ffma, _ = cp.probe_pipe_rate("ffma", 32, 4096)
    do_direct = args.only in ("both", "direct")
    do_cutoff = args.only in ("both", "cutoff")
    # cutoff work accounting (not timed)
    counts = {"useful": 0, "evaluated": 0, "examined": 0}
    stats = None
    if do_cutoff:
        counts = cp.cutoff_pair_counts(ac, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, args.capacity,
                                       workspace=ws)
        stats = cp.cutoff_stats(ws, wc.n_atoms, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, args.capacity)
        if args.shard_map:  # the whole map's pairs: every rank's slab
            counts = dict(zip(("useful", "evaluated", "examined"),
                              (int(v) for v in sum_over_ranks([counts["useful"], counts["evaluated"],
                                                               counts["examined"]], device))))

    sampler = ClockSampler(gpu_id_for(torch, device))
    for _ in range(args.warmup):
        flush.fill_(1)
        if do_direct:
            run_direct()
        flush.fill_(2)
        if do_cutoff:
            run_bin()
            run_map()
    torch.cuda.synchronize()

    def timed_steps(smp):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
        launches0 = lib.cp_launch_count()
        barrier(device)
        torch.cuda.synchronize()
        smp.mark_begin()
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            e = ev[k]
            flush.fill_(k & 0x7F)
            e[0].record(stream)
            if do_direct:
                run_direct()
            e[1].record(stream)
            flush.fill_((k + 64) & 0x7F)
            e[2].record(stream)
            if do_cutoff:
                run_bin()
            e[3].record(stream)
            if do_cutoff:
                run_map()
            e[4].record(stream)
        torch.cuda.synchronize()
        barrier(device)
        t_wall = time.perf_counter() - t_wall0
        smp.mark_end()
        return ev, t_wall, lib.cp_launch_count() - launches0, smp.stop()

    ev, t_wall, launches, clocks = timed_steps(sampler)
    # a slowdown seen on any rank invalidates the attempt: measure once more
    if max_over_ranks([1.0 if clocks_rejected(clocks) else 0.0], device)[0] > 0.0:
        first = clocks
        sampler = ClockSampler(gpu_id_for(torch, device))
        time.sleep(0.5)  # let the sampler start before the steps
        ev, t_wall, launches, clocks = timed_steps(sampler)
        clocks = dict(clocks, remeasured_after={"reasons": first.get("reasons"), "sm_mhz": first.get("sm_mhz")})

    t_direct = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    t_bin = sum(e[2].elapsed_time(e[3]) for e in ev) / 1e3
    t_map = sum(e[3].elapsed_time(e[4]) for e in ev) / 1e3
    # medians of the per-step leg times (ms), beside the means that the rates use
    med_direct = float(np.median([e[0].elapsed_time(e[1]) for e in ev]))
    med_cut = float(np.median([e[2].elapsed_time(e[4]) for e in ev]))
    med_map = float(np.median([e[3].elapsed_time(e[4]) for e in ev]))
    med_bin = float(np.median([e[2].elapsed_time(e[3]) for e in ev]))
    t_direct, t_bin, t_map, t_wall, med_direct, med_cut, med_map, med_bin = max_over_ranks(
        [t_direct, t_bin, t_map, t_wall, med_direct, med_cut, med_map, med_bin], device)
    t_direct, t_bin, t_map = (max(t, 1e-12) for t in (t_direct, t_bin, t_map))
    K = args.steps
    # counts are the whole map's in --shard-map mode, one rank's otherwise
    cmul = 1 if args.shard_map else world
    direct_rate = float(wd_full.n_pairs) * job * K / t_direct
    t_cut = t_bin + t_map
    points_rate = float(wc_full.n_points) * job * K / t_cut

    f_mhz = clocks.get("sm_mhz") or 2070.0
    clock_basis = "median SM clock sampled during the timed steps" if clocks.get("sm_mhz") else "max SM clock"
    roof = Roofline(r_mufu, r_ffma, n_sm, f_mhz, clock_basis)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    hbm_basis = "of measured" if "hbm_gbs" in peaks else "of fallback"

    # the cutoff leg again as one captured CUDA graph (binning's five launches
    # and the map replayed without per-launch host overhead)
    t_graph_cut = None
    if do_cutoff:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            gs = torch.cuda.current_stream().cuda_stream
            call(lib.cp_bin_atoms(ac.data_ptr(), wc.n_atoms, *gc, *cut, ws.data_ptr(), ws_bytes, gs), "cp_bin_atoms")
            call(lib.cp_cutoff_map(ac.data_ptr(), wc.n_atoms, *gc, *cut, ws.data_ptr(), ws_bytes, Vc.data_ptr(), gs),
                 "cp_cutoff_map")
        graph.replay()
        torch.cuda.synchronize()
        tg = []
        for _ in range(max(3, min(args.steps, 20))):
            flush.fill_(5)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            tg.append(e0.elapsed_time(e1))
        t_graph_cut = float(np.mean(tg)) / 1e3
        del graph

    # every other workload, one at a time (3 warm-ups, 10 timed runs, L2
    # flushed before each); not part of the step
    secondary = None
    if not args.no_secondary:
        sec_sampler = ClockSampler(gpu_id_for(torch, device))
        sec_sampler.mark_begin()
        secondary = measure_secondary(cp, lib, torch, device, stream, flush, roof, hbm_peak, hbm_basis,
                                      do_direct, do_cutoff, args.capacity, {args.cutoff_workload: wc_full})
        sec_sampler.mark_end()
        secondary["clocks"] = sec_sampler.stop()

    # multilevel long-range part on the 200^3 / 100k-atom cutoff workload
    # (reported beside the step, not part of it)
    msm = None
    if do_cutoff and not args.no_msm:
        msm = measure_msm(cp, lib, torch, device, stream, flush, args, roof, call)
    status = cp.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status:#x} after the timed steps")

    # end to end through the public API with host buffers ---------------------
    n_e2e = max(3, min(K, 5))
    t_e2e_d = t_e2e_c = float("nan")
    if not args.no_e2e:
        host_atoms_d = torch.from_numpy(wd.atoms).pin_memory()
        host_out_d = torch.empty(Vd.shape, dtype=torch.float32, pin_memory=True)
        host_atoms_c = torch.from_numpy(wc.atoms).pin_memory()
        host_out_c = torch.empty(Vc.shape, dtype=torch.float32, pin_memory=True)
        t_e2e_d, t_e2e_c = e2e_times(cp, wd, wc, Vd, Vc, ws, host_atoms_d, host_out_d, host_atoms_c, host_out_c,
                                     n_e2e, args.capacity, do_direct, do_cutoff)
        t_e2e_d, t_e2e_c = max_over_ranks([t_e2e_d, t_e2e_c], device)

    # --shard-map: the gather of the slabs to rank 0 (after the steps, timed once)
    gather = None
    if args.shard_map and world > 1:
        from direct_coulomb_summation_gb300 import shard

        gather = {}
        for key, V, w, align in (("direct", Vd, wd_full, 1), ("cutoff", Vc, wc_full, 8)):
            barrier(device)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            shard.gather_slabs(V, w.shape, align, dst=0)
            torch.cuda.synchronize()
            gather["ms_" + key] = max_over_ranks([1e3 * (time.perf_counter() - t0)], device)[0]
        gather["bytes"] = {"direct": wd_full.n_points * 4, "cutoff": wc_full.n_points * 4}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # CPU baseline: the oracle on this host's cores, bounded samples
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        threads = host_threads()
        rate, n_pts, dt = oracle_direct_rate(wd_full, args.cpu_seconds, threads)
        crate, c_pts, cdt = oracle_cutoff_rate(wc_full, args.cpu_seconds / 2, threads)
        srate, s_pts, sdt = oracle_direct_rate(wd_full, args.cpu_seconds / 4, 1)
        cpu = {"value": rate, "unit": "pair evals/s", "cores": threads, "kind": "oracle",
               "sample": f"fp64 direct sum at {n_pts} seeded grid points of the {tuple(wd.shape)} grid x "
                         f"{wd.n_atoms} atoms ({dt:.1f} s)",
               "single_core": {"value": srate, "unit": "pair evals/s", "cores": 1,
                               "sample": f"the same sum at {s_pts} points on one thread ({sdt:.1f} s)"},
               "cutoff": {"value": crate, "unit": "grid points/s",
                          "sample": f"fp64 binned cutoff sum at {c_pts} seeded points of the {tuple(wc.shape)} "
                                    f"grid ({cdt:.1f} s)"}}

    traffic = traffic_from_profile("direct_kernel", "direct_coulomb_summation_gb300/csrc/cp_direct.cu",
                                   args.direct_workload)
    traffic_map = traffic_from_profile("cutoff_brick_kernel", "direct_coulomb_summation_gb300/csrc/cp_cutoff.cu",
                                       args.cutoff_workload)
    rd = roof.direct(direct_rate, world)
    useful_rate = counts["useful"] * cmul * K / t_map
    L = cp.cutoff_layout(wc.n_atoms, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, args.capacity)
    bin_bytes = bin_bytes_of(L, wc.n_atoms, args.capacity)
    line = {
        "metric": METRIC,
        "value": direct_rate,
        "unit": "pair evals/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * (t_direct + t_cut) / K,
        "higher_is_better": True,
        "scaling": "strong" if args.shard_map else "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config_dict(wd_full, wc_full, args.capacity, world if args.shard_map else 0),
        "roofline": {
            "bound": "alu",
            "kernel": "direct_kernel (cp_direct)",
            "workload": wd.description,
            "achieved": rd["achieved"],
            "peak": rd["peak"],
            "unit": "pair evals/s",
            "frac": rd["frac"],
            "traffic": traffic,
            "peak_basis": f"{n_sm} SMs x {roof.direct_split:.1f} pairs/clk/SM x {f_mhz:.0f} MHz ({clock_basis}): "
                          f"the pair (1 rsqrt, 3 FP32 ops) with its rsqrt shared between the SFU "
                          f"({r_mufu:.2f}/clk/SM measured) and the FMA pipe (magic-constant estimate + two Newton "
                          f"steps, 6 FP32 ops; FFMA {r_ffma:.1f} lanes/clk/SM measured) at the best share "
                          f"{roof.f_split:.2f}, (1 - f)/R_sfu = (3 + 6f)/R_fp32",
            "peak_sfu_only": rd["peak_sfu_only"],
            "frac_sfu_only": rd["frac_sfu_only"],
            "sfu_only_basis": f"{n_sm} SMs x {roof.direct_sfu:.2f} pairs/clk/SM = min(SFU rsqrt {r_mufu:.2f}, "
                              f"FFMA {r_ffma:.1f}/3, issue 128/4): the scope table's bound for rsqrt on the SFU "
                              f"alone, which the kernel exceeds by moving a share of the rsqrts to the FMA pipe",
        },
        "direct": {
            "config": CONFIG_NUMBER.get(args.direct_workload),
            "pair_evals_per_s": direct_rate,
            "grid_points_per_s": float(wd_full.n_points) * job * K / t_direct,
            "ms": 1e3 * t_direct / K,
            "ms_median": med_direct if do_direct else None,
            "plan": list(cp.direct_plan(wd.n_atoms, wd.shape)),
        },
        "cutoff": {
            "config": CONFIG_NUMBER.get(args.cutoff_workload),
            "capacity": args.capacity,
            "grid_points_per_s": points_rate,
            "useful_pairs_per_s": counts["useful"] * cmul * K / t_cut,
            "evaluated_pairs_per_s": counts["evaluated"] * cmul * K / t_cut,
            "examined_pairs_per_s": counts["examined"] * cmul * K / t_cut,
            "pairs_per_step": counts,
            "evaluated_per_useful": counts["evaluated"] / counts["useful"] if counts["useful"] else None,
            "binning_stats": stats,
            "overflow_atoms": None if (stats is None or args.capacity == 0) else stats["n_overflow"],
            "binning_note": "capacity 0 has no fixed slots: every atom is read from its bin's contiguous run, so "
                            "n_overflow counts all binned atoms" if args.capacity == 0 else
                            "n_overflow = atoms past the fixed slots, read by the overflow sweep",
            "ms": 1e3 * t_cut / K,
            "ms_median": med_cut if do_cutoff else None,
            "ms_binning": 1e3 * t_bin / K,
            "ms_binning_median": med_bin if do_cutoff else None,
            "ms_map": 1e3 * t_map / K,
            "ms_map_median": med_map if do_cutoff else None,
            "ms_as_cuda_graph": None if t_graph_cut is None else 1e3 * t_graph_cut,
            "roofline_map": dict(
                roof.cutoff(useful_rate, world), bound="alu", kernel="cutoff_brick_kernel (cp_cutoff_map)",
                traffic=traffic_map,
                peak_basis=f"{n_sm} SMs x {roof.useful:.2f} useful pairs/clk/SM = min(SFU {r_mufu:.2f}, "
                           f"FFMA {r_ffma:.1f}/11) x {f_mhz:.0f} MHz",
                tight_basis=f"min(SFU {r_mufu:.2f}, 128 issue/8) = {roof.useful_tight:.1f} useful pairs/clk/SM"),
            "roofline_binning": {
                "bound": "hbm", "achieved": bin_bytes * world * K / t_bin / 1e9, "peak": hbm_peak * world,
                "unit": "GB/s", "frac": bin_bytes * K / t_bin / 1e9 / hbm_peak,
                "traffic": traffic_from_profile("binning", "direct_coulomb_summation_gb300/csrc/cp_cutoff.cu",
                                                args.cutoff_workload),
                "algorithmic_bytes": bin_bytes, "peak_basis": f"hbm_gbs {hbm_basis}",
            },
        },
        "secondary": secondary,
        "shard_gather": gather,
        "msm": msm,
        "cpu_baseline": cpu,
        "e2e": {
            "value": float(wd_full.n_pairs) * job / t_e2e_d,
            "unit": "pair evals/s",
            "h2d_bytes_per_step": int(wd.atoms.nbytes),
            "d2h_bytes_per_step": int(Vd.numel() * 4),
            "cutoff_grid_points_per_s": float(wc_full.n_points) * job / t_e2e_c,
            "cutoff_h2d_bytes": int(wc.atoms.nbytes),
            "cutoff_d2h_bytes": int(Vc.numel() * 4),
            "how": "public Python API with pinned host atoms in, host V out; wall clock per call incl. copies",
        },
        "gpu_launches": int(launches),
        "clocks": clocks,
        "wall_ms_per_step": 1e3 * t_wall / K,
        "device": props.name,
    }
    if not do_cutoff:
        line["cutoff"] = None
    if not do_direct:
        for key in ("value", "roofline", "direct"):
            line[key] = None
    if args.no_e2e:
        line["e2e"] = None
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _timed_runs(torch, stream, flush, fns, reps=10, warm=3):
    """The pwwt.cn article's protocol: warm-ups, then `reps` runs with L2
    flushed before each; `fns` run back to back and each is timed with CUDA
    events on `stream`.  Returns per-fn lists of ms."""
    for _ in range(warm):
        for fn in fns:
            fn()
    out = [[] for _ in fns]
    for r in range(reps):
        flush.fill_(r & 0x7F)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
        ev[0].record(stream)
        for i, fn in enumerate(fns):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        for i in range(len(fns)):
            out[i].append(ev[i].elapsed_time(ev[i + 1]))
    return out


def measure_secondary(cp, lib, torch, device, stream, flush, roof, hbm_peak, hbm_basis, do_direct, do_cutoff,
                      head_capacity, workloads_done=None):
    sh = stream.cuda_stream
    res = {"protocol": "3 warm-ups, 10 timed runs each, 256 MiB L2 flush before each run, CUDA events; "
                       "not part of the timed steps", "direct": {}, "cutoff": {}}

    def call(rc, where):
        if rc != 0:
            raise cp.CpError(rc, where)

    if do_direct:
        for name in SECONDARY_DIRECT:
            w = make_workload(name)
            a = torch.from_numpy(w.atoms).to(device)
            V = torch.empty((w.shape[2], w.shape[1], w.shape[0]), dtype=torch.float32, device=device)
            g = cp._grid(w.shape, w.origin, w.h)
            (ts,) = _timed_runs(torch, stream, flush, [
                lambda: call(lib.cp_direct(a.data_ptr(), w.n_atoms, *g, V.data_ptr(), sh), "cp_direct")])
            mean = float(np.mean(ts))
            rate = w.n_pairs / (mean * 1e-3)
            rd = roof.direct(rate)
            res["direct"][name] = {
                "config": CONFIG_NUMBER[name], "workload": w.description, "grid": list(w.shape), "atoms": w.n_atoms,
                "pairs": w.n_pairs, "ms": mean, "ms_median": float(np.median(ts)), "pair_evals_per_s": rate,
                "grid_points_per_s": w.n_points / (mean * 1e-3), "roofline_frac": rd["frac"],
                "frac_sfu_only": rd["frac_sfu_only"], "plan": list(cp.direct_plan(w.n_atoms, w.shape))}
            del a, V
    if do_cutoff:
        cache = dict(workloads_done or {})
        for name, K in SECONDARY_CUTOFF:
            if name == CUTOFF_WL and K == head_capacity:
                continue
            if name not in cache:
                cache[name] = make_workload(name)
            w = cache[name]
            a = torch.from_numpy(w.atoms).to(device)
            V = torch.empty((w.shape[2], w.shape[1], w.shape[0]), dtype=torch.float32, device=device)
            nbytes = cp.cutoff_workspace_bytes(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, K)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
            g = cp._grid(w.shape, w.origin, w.h)
            cut = [float(np.float32(w.cutoff)), float(np.float32(w.bin_size)), K]
            counts = cp.cutoff_pair_counts(a, w.shape, w.origin, w.h, w.cutoff, w.bin_size, K, workspace=ws)
            stats = cp.cutoff_stats(ws, w.n_atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, K)
            tb, tm = _timed_runs(torch, stream, flush, [
                lambda: call(lib.cp_bin_atoms(a.data_ptr(), w.n_atoms, *g, *cut, ws.data_ptr(), nbytes, sh),
                             "cp_bin_atoms"),
                lambda: call(lib.cp_cutoff_map(a.data_ptr(), w.n_atoms, *g, *cut, ws.data_ptr(), nbytes,
                                               V.data_ptr(), sh), "cp_cutoff_map")])
            mb, mm = float(np.mean(tb)), float(np.mean(tm))
            L = cp.cutoff_layout(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, K)
            bb = bin_bytes_of(L, w.n_atoms, K)
            entry = {
                "config": CONFIG_NUMBER[name], "workload": w.description, "capacity": K,
                "layout": "contiguous bin-sorted runs" if K == 0 else f"{K} fixed slots per bin + overflow list",
                "ms": mb + mm, "ms_median": float(np.median(np.asarray(tb) + np.asarray(tm))),
                "ms_binning": mb, "ms_map": mm, "ms_map_median": float(np.median(tm)),
                "grid_points_per_s": w.n_points / ((mb + mm) * 1e-3),
                "useful_pairs_per_s": counts["useful"] / ((mb + mm) * 1e-3),
                "pairs": counts, "evaluated_per_useful": counts["evaluated"] / max(counts["useful"], 1),
                "binning_stats": stats,
                "overflow_atoms": None if K == 0 else stats["n_overflow"],
                "roofline_map": roof.cutoff(counts["useful"] / (mm * 1e-3)),
                "roofline_binning": {"bound": "hbm", "achieved": bb / (mb * 1e-3) / 1e9, "peak": hbm_peak,
                                     "unit": "GB/s", "frac": bb / (mb * 1e-3) / 1e9 / hbm_peak,
                                     "algorithmic_bytes": bb, "peak_basis": f"hbm_gbs {hbm_basis}"},
            }
            res["cutoff"][f"{name}/capacity_{K}"] = entry
            del a, V, ws
    torch.cuda.synchronize()
    return res


def measure_msm(cp, lib, torch, device, stream, flush, args, roof, call):
    """cp_msm_longrange adding V_long to the 200^3 / 100k-atom cutoff map."""
    sh = stream.cuda_stream
    w = make_workload("cutoff_uniform")
    a = torch.from_numpy(w.atoms).to(device)
    V = torch.empty((w.shape[2], w.shape[1], w.shape[0]), dtype=torch.float32, device=device)
    g = cp._grid(w.shape, w.origin, w.h)
    cut = [float(np.float32(w.cutoff)), float(np.float32(w.bin_size)), 0]
    nbytes = cp.cutoff_workspace_bytes(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    lo, hi = cp.atom_bounds(a)
    dom = (cp._vec3(lo), cp._vec3(hi))
    h0 = float(np.float32(args.msm_lattice))
    ML = cp.msm_layout(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, h0, (lo, hi))
    mws = torch.empty(int(ML.total_bytes), dtype=torch.uint8, device=device)

    def run_cut():
        call(lib.cp_cutoff(a.data_ptr(), w.n_atoms, *g, *cut, ws.data_ptr(), nbytes, V.data_ptr(), sh), "cp_cutoff")

    def run_msm():
        call(lib.cp_msm_longrange(a.data_ptr(), w.n_atoms, *g, *dom, cut[0], h0, mws.data_ptr(),
                                  int(ML.total_bytes), V.data_ptr(), 1, sh), "cp_msm_longrange")

    c_launch0 = lib.cp_launch_count()
    run_cut()
    launches_cut = lib.cp_launch_count() - c_launch0
    m_launch0 = lib.cp_launch_count()
    tc, tm = _timed_runs(torch, stream, flush, [run_cut, run_msm], reps=max(3, min(args.steps, 20)))
    n_calls = 3 + max(3, min(args.steps, 20))
    levels = int(ML.levels)
    nodes = [int(ML.n[l][0]) * int(ML.n[l][1]) * int(ML.n[l][2]) for l in range(levels)]
    # algorithmic FMAs of the lattice cutoffs: every node of every level
    # below the top times the stencil's taps, plus the dense top level
    fma = sum(nodes[:-1]) * int(ML.taps) + nodes[-1] ** 2
    ms_l, ms_c = float(np.median(tm)), float(np.median(tc))
    return {"workload": w.description, "lattice_h": h0, "levels": levels, "nodes": nodes,
            "stencil_taps": int(ML.taps), "ms_longrange": ms_l,
            "launches_per_call": int((lib.cp_launch_count() - m_launch0) // n_calls - launches_cut),
            "lattice_cutoff_fma_per_call": fma, "ms_map": ms_c + ms_l,
            "grid_points_per_s_map": w.n_points / (1e-3 * (ms_c + ms_l)),
            "fp32_fma_per_s_longrange": fma / (1e-3 * ms_l),
            "frac_of_fp32_fma": fma / (1e-3 * ms_l) / (roof.r_ffma * roof.sm_clk),
            "basis": "the whole cp_msm_longrange call (cell sort, anterpolation, restriction, lattice cutoffs, "
                     "prolongation, interpolation) against the FP32 FMA rate for its lattice-cutoff FMAs alone; "
                     "ms_map adds the cutoff map of the same grid (binning + short-range map, capacity 0): the "
                     "multilevel approximation of the full direct sum on this grid"}


def run_compare(args):
    """The pwwt.cn chapter-18 article's five-way comparison on its own case
    (z-index 10 plane of a 100x100x50 grid at 0.5 A, 10 000 atoms): the
    sequential CPU sum (the fp64 oracle on one core), the GPU scatter, gather,
    coarsened and coarsened + coalesced kernels, and this library's direct
    kernel; plus the notes' 27-bin hard-cutoff kernel against the brick map on
    the 200^3 / 100k-atom cutoff workload.  3 warm-ups and 10 timed runs each,
    L2 flushed before every run, CUDA events; one JSON line."""
    import torch

    import direct_coulomb_summation_gb300 as cp
    import oracle
    import workloads

    rank, world, local = env_rank()
    if rank != 0:
        return 0
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def timed(fn, reps=10, warm=3):
        for _ in range(warm):
            fn()
        ts = []
        for _ in range(reps):
            flush.fill_(3)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.mean(ts)), float(np.median(ts))

    w = workloads.make("direct_plane")
    a = torch.from_numpy(w.atoms).to(device)
    V = torch.empty((w.shape[2], w.shape[1], w.shape[0]), dtype=torch.float32, device=device)
    t0 = time.perf_counter()
    oracle.direct(w.atoms, w.shape, w.origin, w.h, threads=1, with_bound=False)
    seq_ms = 1e3 * (time.perf_counter() - t0)
    res = {"sequential (fp64 oracle, 1 core)": {"ms": seq_ms}}
    for name in ("scatter", "gather", "coarsen", "coalesce"):
        mean, med = timed(lambda: cp.direct_variant(name, a, w.shape, w.origin, w.h, out=V))
        res[f"gpu {name}"] = {"ms": mean, "ms_median": med}
    mean, med = timed(lambda: cp.direct(a, w.shape, w.origin, w.h, out=V))
    res["gpu cp_direct (this library)"] = {"ms": mean, "ms_median": med}
    # the same call captured once as a CUDA graph and replayed: on a map this
    # small, the difference is the per-launch host and launch overhead
    graph = torch.cuda.CUDAGraph()
    cp.direct(a, w.shape, w.origin, w.h, out=V)  # plans and sets kernel attributes before capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        cp.direct(a, w.shape, w.origin, w.h, out=V)
    mean, med = timed(graph.replay)
    res["gpu cp_direct (this library), replayed as a CUDA graph"] = {"ms": mean, "ms_median": med}
    for v in res.values():
        v["pair_evals_per_s"] = w.n_pairs / (v["ms"] * 1e-3)
        v["speedup_vs_sequential"] = seq_ms / v["ms"]

    wc = workloads.make("cutoff_uniform")
    ac = torch.from_numpy(wc.atoms).to(device)
    Vc = torch.empty((wc.shape[2], wc.shape[1], wc.shape[0]), dtype=torch.float32, device=device)
    ws = torch.empty(max(cp.cutoff_workspace_bytes(wc.n_atoms, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, 0),
                         int(cp.library().cp_cutoff27_workspace_bytes(wc.n_atoms, *cp._grid(wc.shape, wc.origin, wc.h),
                                                                      float(wc.cutoff)))),
                     dtype=torch.uint8, device=device)
    cut = {}
    mean, med = timed(lambda: cp.cutoff27(ac, wc.shape, wc.origin, wc.h, wc.cutoff, workspace=ws, out=Vc))
    cut["27-bin hard cutoff (bins of edge c, one thread per point)"] = {"ms": mean, "ms_median": med}
    mean, med = timed(lambda: cp.cutoff(ac, wc.shape, wc.origin, wc.h, wc.cutoff, wc.bin_size, 0, workspace=ws,
                                        out=Vc))
    cut["brick map with switched term (this library, binning included)"] = {"ms": mean, "ms_median": med}
    for v in cut.values():
        v["grid_points_per_s"] = wc.n_points / (v["ms"] * 1e-3)
    print(json.dumps({"compare": "strategies of the pages on their own workloads", "device": torch.cuda.get_device_name(),
                      "direct_workload": w.description, "direct": res,
                      "cutoff_workload": wc.description, "cutoff": cut,
                      "protocol": "3 warm-ups, 10 timed runs, 256 MiB L2 flush before each, CUDA events"}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-msm", action="store_true", help="skip the multilevel long-range measurement")
    ap.add_argument("--msm-lattice", type=float, default=2.0, help="finest lattice spacing of the long-range part")
    ap.add_argument("--only", choices=["both", "direct", "cutoff"], default="both",
                    help="time one leg only (for profiling; the JSON line then covers that leg)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--shard-map", action="store_true",
                    help="the ranks share one map as z-slabs (strong scaling) instead of one copy each")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the per-workload timings after the steps (for profiling)")
    ap.add_argument("--direct-workload", choices=["direct_plane", "direct_3d", "direct_protein"], default=DIRECT_WL,
                    help="direct workload of the step (the default is the headline; others for profiling)")
    ap.add_argument("--cutoff-workload", choices=["cutoff_uniform", "cutoff_large"], default=CUTOFF_WL,
                    help="cutoff workload of the step (the default is the headline; others for profiling)")
    ap.add_argument("--compare", action="store_true",
                    help="time the pages' own strategies against this library (one JSON line) and exit")
    ap.add_argument("--capacity", type=int, choices=[0, 8, 16], default=CAPACITY_DEFAULT,
                    help="bin capacity of the cutoff leg (0 = contiguous bin-sorted runs, no fixed slots)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.compare:
        return run_compare(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
