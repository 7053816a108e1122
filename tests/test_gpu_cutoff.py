"""GPU parity of the cutoff map (binning + brick kernel + overflow sweep)
against the fp64 oracle, within |V_gpu - V_ref| <= 2e-4 * sum_{r<c} |q|/r."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from gpu_util import assert_within_bound, flat_index, to_dev

pytestmark = pytest.mark.gpu


def _run(w, c, b, K=16, **kw):
    V = cp.cutoff(to_dev(w.atoms), w.shape, w.origin, w.h, c, b, capacity=K, **kw)
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    return V


@pytest.mark.parametrize("K", [0, 8, 16])
@pytest.mark.parametrize("seed,n,shape,h,origin,c,b", [
    (301, 1500, (24, 20, 17), 0.5, (0.0, 0.0, 0.0), 3.0, 1.0),
    (302, 900, (19, 23, 16), 0.4, (-2.1, 0.7, 3.3), 2.5, 1.3),     # bricks not aligned with bins
    (303, 2500, (33, 9, 12), 0.5, (1.0, -4.0, 0.5), 4.0, 4.0),     # ragged bricks, big bins
    (304, 700, (16, 16, 1), 0.5, (0.0, 0.0, 5.0), 2.0, 0.75),      # single plane
    (305, 3000, (21, 9, 30), 0.3, (10.0, -5.0, 0.25), 1.9, 0.55),
    (306, 1200, (14, 11, 9), 1.5, (0.5, 0.0, -1.0), 2.0, 0.8),      # grid spacing above the bin size
])
def test_cutoff_small_full_grid(K, seed, n, shape, h, origin, c, b):
    w = workloads.random_case(seed, n, shape, h=h, origin=origin, margin=c + 1.0)
    V = _run(w, c, b, K)
    ref, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    assert_within_bound(V.cpu().numpy(), ref, bound, w.name)


@pytest.mark.parametrize("K", [0, 8, 16])
def test_cutoff_all_atoms_in_one_bin(K):
    """Every atom in one bin: capacity overflow for every atom past K."""
    rng = np.random.default_rng(5)
    shape, h, c, b = (24, 24, 24), 0.5, 3.0, 1.0
    n = 600
    atoms = np.empty((n, 4), dtype=np.float32)
    atoms[:, :3] = (6.0 + rng.uniform(0.05, 0.45, size=(n, 3))).astype(np.float32)
    atoms[:, 3] = rng.uniform(-1, 1, size=n).astype(np.float32)
    w = workloads.Workload("one_bin", atoms, shape, (0.0, 0.0, 0.0), h)
    V = _run(w, c, b, K)
    ref, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    assert_within_bound(V.cpu().numpy(), ref, bound, "one bin")


def test_cutoff_atoms_outside_and_nonfinite():
    w = workloads.random_case(7, 800, (16, 16, 16), margin=12.0)  # many atoms far outside
    extra = np.array([[np.nan, 1, 1, 1], [np.inf, 1, 1, 1], [1e30, 0, 0, 1]], dtype=np.float32)
    atoms = np.concatenate([w.atoms, extra])
    c, b = 2.5, 1.0
    V = cp.cutoff(to_dev(atoms), w.shape, w.origin, w.h, c, b)
    torch.cuda.synchronize()
    ref, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    assert_within_bound(V.cpu().numpy(), ref, bound, "outside")


def test_cutoff_zero_atoms():
    V = cp.cutoff(torch.zeros((0, 4), dtype=torch.float32, device="cuda"), (9, 9, 9), (0, 0, 0), 0.5, 2.0, 1.0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(V).item() == 0


def test_cutoff_large_c_tends_to_direct():
    """With every pair inside the cutoff, cutoff + (15/(8c)) sum q = direct + O(r^2/c^3)."""
    w = workloads.random_case(8, 1200, (20, 16, 12), margin=1.0)
    c = 200.0
    Vc = _run(w, c, 64.0)
    Vd = cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    qsum = float(w.atoms[:, 3].astype(np.float64).sum())
    _, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    diff = (Vc.double() + 15.0 / (8.0 * c) * qsum - Vd.double()).cpu().numpy().reshape(-1)
    rmax = 30.0
    lim = (5 / 4) * rmax**2 / c**3 * np.abs(w.atoms[:, 3]).sum() + 4e-4 * bound
    assert np.all(np.abs(diff) <= lim)


def test_cutoff_workspace_reuse_and_determinism():
    w = workloads.random_case(9, 4000, (40, 32, 24), margin=3.0)
    c, b = 3.0, 1.0
    need = cp.cutoff_workspace_bytes(4000, w.shape, w.origin, w.h, c, b)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    a = to_dev(w.atoms)
    v1 = cp.cutoff(a, w.shape, w.origin, w.h, c, b, workspace=ws).clone()
    v2 = cp.cutoff(a, w.shape, w.origin, w.h, c, b, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(v1, v2)


def test_cutoff_host_buffers_match_device():
    w = workloads.random_case(10, 900, (20, 12, 6), margin=1.0)
    vh = cp.cutoff(w.atoms, w.shape, w.origin, w.h, 2.0, 1.0)
    vd = cp.cutoff(to_dev(w.atoms), w.shape, w.origin, w.h, 2.0, 1.0)
    torch.cuda.synchronize()
    assert not vh.is_cuda and torch.equal(vh, vd.cpu())


def _benchmark_call(w, K):
    """The cutoff map as bench.py times it: cp_bin_atoms then cp_cutoff_map
    through the C ABI on one caller-owned workspace, c and b from the
    workload (12 A, 4 A)."""
    lib = cp.library()
    a = to_dev(w.atoms)
    V = torch.full((w.shape[2], w.shape[1], w.shape[0]), float("nan"), device="cuda")
    nbytes = cp.cutoff_workspace_bytes(w.n_atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, K)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    g = cp._grid(w.shape, w.origin, w.h)
    cut = (float(np.float32(w.cutoff)), float(np.float32(w.bin_size)), K)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.cp_bin_atoms(a.data_ptr(), w.n_atoms, *g, *cut, ws.data_ptr(), nbytes, s) == 0
    assert lib.cp_cutoff_map(a.data_ptr(), w.n_atoms, *g, *cut, ws.data_ptr(), nbytes, V.data_ptr(), s) == 0
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    return V


@pytest.mark.parametrize("K", [0, 16])
def test_cutoff_uniform_workload_sampled(K):
    """100 000 atoms, 200^3 grid, c = 12 A, 4 A bins (capacity 0 is the
    benchmarked layout): full map on the GPU in the benchmark's two calls,
    4096 seeded points by the brute-force oracle."""
    w = workloads.make("cutoff_uniform")
    V = _benchmark_call(w, K)
    pts = workloads.sample_points(w.shape, 4096, seed=4097)
    ref, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, w.cutoff, points=pts)
    got = V.reshape(-1)[torch.from_numpy(flat_index(w.shape, pts)).cuda()].cpu().numpy()
    assert_within_bound(got, ref, bound, w.name)
    assert torch.isfinite(V).all()


@pytest.mark.parametrize("K", [0, 16])
def test_cutoff_uniform_workload_brick_layers(K):
    """Whole brick layers of the 200^3 map (the first, a middle and the last
    8 planes: every brick of them, edges included) against the binned oracle
    at every point."""
    w = workloads.make("cutoff_uniform")
    V = _benchmark_call(w, K)
    nx, ny, nz = w.shape
    for z0 in (0, 96, nz - 8):
        ij = np.stack(np.meshgrid(np.arange(nx), np.arange(ny), indexing="xy"), -1).reshape(-1, 2)
        pts = np.concatenate([np.column_stack([ij, np.full(len(ij), z)]) for z in range(z0, z0 + 8)])
        ref, bound = oracle.cutoff_binned(w.atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, points=pts)
        got = V.reshape(-1)[torch.from_numpy(flat_index(w.shape, pts)).cuda()].cpu().numpy()
        assert_within_bound(got, ref, bound, f"{w.name} planes {z0}..{z0 + 7}")


@pytest.mark.parametrize("K", [0, 16])
def test_cutoff_large_workload_sampled(K):
    """800 000 atoms (30 % in Gaussian clusters), 400^3 grid, c = 12 A, 4 A
    bins, in the benchmark's two calls: 4096 seeded points by the binned
    oracle (bit-identical to brute force by its pins)."""
    w = workloads.make("cutoff_large")
    V = _benchmark_call(w, K)
    pts = workloads.sample_points(w.shape, 4096, seed=4098)
    ref, bound = oracle.cutoff_binned(w.atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, points=pts)
    got = V.reshape(-1)[torch.from_numpy(flat_index(w.shape, pts)).cuda()].cpu().numpy()
    assert_within_bound(got, ref, bound, w.name)
    assert torch.isfinite(V).all()


def _pairs_within(w, c, rel):
    """Pairs (grid point, atom) with r^2 < c^2 (1 + rel), in fp64 from the same fp32 inputs."""
    a = w.atoms[:, :3].astype(np.float64)
    o = np.asarray([np.float32(v) for v in w.origin], dtype=np.float64)
    h = float(np.float32(w.h))
    ijk = workloads.grid_points(w.shape).astype(np.float64)
    lim = float(np.float32(c)) ** 2 * (1.0 + rel)
    total = 0
    for s in range(0, ijk.shape[0], 2048):
        g = o + ijk[s:s + 2048] * h
        d2 = ((g[:, None, :] - a[None, :, :]) ** 2).sum(-1)
        total += int(np.count_nonzero(d2 < lim))
    return total


@pytest.mark.parametrize("K", [0, 16])
@pytest.mark.parametrize("seed,n,shape,h,origin,c,b", [
    (321, 1500, (24, 20, 17), 0.5, (0.0, 0.0, 0.0), 6.0, 2.0),
    (322, 1200, (19, 23, 16), 0.4, (-2.1, 0.7, 3.3), 3.0, 1.3),
    (323, 2000, (33, 9, 12), 0.5, (1.0, -4.0, 0.5), 12.0, 4.0),   # the benchmark's c and bin size
])
def test_cutoff_useful_pairs_exact(K, seed, n, shape, h, origin, c, b):
    """The counting variant of the brick traversal (behind the useful-pair rate the
    benchmark reports) counts the pairs whose fp32 r^2 is below c^2 at stored
    points.  That count must fall between the fp64 counts with c^2 narrowed and
    widened by 2e-6 (the fp32 rounding of r^2 and of the grid coordinates), and
    the traversal's evaluated and examined counts must bound it."""
    w = workloads.random_case(seed, n, shape, h=h, origin=origin, margin=c + 1.0)
    counts = cp.cutoff_pair_counts(to_dev(w.atoms), w.shape, w.origin, w.h, c, b, capacity=K)
    lo, hi = _pairs_within(w, c, -2e-6), _pairs_within(w, c, 2e-6)
    assert lo <= counts["useful"] <= hi, (counts, lo, hi)
    assert counts["useful"] <= counts["evaluated"] <= counts["examined"]


def _boundary_atoms(origin, h, c, rng):
    """Atoms at distance c(1 + eps) from a corner of consumer-warp sub-boxes
    (8 x 4 x 4 points of an 8x8x8 brick): along the sub-box diagonal from its
    low corner (that corner is then the sub-box point farthest from the atom,
    so the atom is within c of the whole sub-box iff c(1 + eps) < c), and
    beyond its high corner (the nearest point).  eps spans -1e-3 .. 1e-3,
    down to a few fp32 ulps either side of c."""
    o = np.asarray(origin, dtype=np.float64)
    atoms = []
    for brick in ((0, 0, 0), (1, 1, 1), (2, 1, 0)):
        for w in range(4):
            lo = o + h * np.array([8 * brick[0], 8 * brick[1] + 4 * (w & 1), 8 * brick[2] + 4 * (w >> 1)])
            hi = lo + h * np.array([7.0, 3.0, 3.0])
            diag = (hi - lo) / np.linalg.norm(hi - lo)
            for eps in (-1e-3, -1e-5, -1e-6, -1e-7, 0.0, 1e-7, 1e-6, 1e-5, 1e-3):
                R = c * (1.0 + eps)
                atoms.append(list(lo + R * diag) + [rng.uniform(-1, 1)])
                atoms.append(list(hi + R * np.ones(3) / np.sqrt(3.0)) + [rng.uniform(-1, 1)])
    return np.asarray(atoms, dtype=np.float32)


@pytest.mark.parametrize("K", [0, 16])
@pytest.mark.parametrize("offset,h", [(0.0, 0.5), (5000.0, 0.37)])
def test_cutoff_atoms_on_the_full_boundary(K, offset, h):
    """An atom just inside c of a whole sub-box takes the moments path (q/r per
    pair, -q g(r) from the sub-box's charge moments), one just outside it the
    per-pair switched term.  At every point the map must match the brute-force
    oracle within the bound -- exactly 0 where no atom is strictly inside c --
    on a grid at the coordinate origin and on one 5000 A out (differences
    relative to the grid origin)."""
    rng = np.random.default_rng(777)
    c, b = 3.0, 1.0
    origin = (offset + 0.0, -offset, offset / 2) if offset else (0.0, 0.0, 0.0)
    origin = tuple(float(np.float32(v)) for v in origin)
    atoms = _boundary_atoms(origin, float(np.float32(h)), c, rng)
    w = workloads.Workload("full_boundary", atoms, (24, 24, 24), origin, h)
    V = _run(w, c, b, K)
    ref, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    assert (np.asarray(bound) == 0).any()  # points no atom reaches: V must be exactly 0 there
    assert_within_bound(V.cpu().numpy(), ref, bound, f"full boundary K={K} offset={offset}")
