"""Parity of the multilevel long-range path (cp_msm_longrange) with the fp64
oracle (oracle/msm.py), through the C ABI.

Tolerances.  The GPU runs the oracle's steps in fp32: every lattice value is
a sum of at most a few thousand products (7,123 stencil taps at c/h0 = 6),
each rounded once, so its error is a small multiple of 6e-8 times the sum
of the magnitudes it adds, far below the method's own error (about 1e-4 of
B(x) = sum_a |q_a| g_c(|x - r_a|) at c/h0 = 6).  The tests allow
|V_gpu - V_oracle| <= 1e-5 B(x): ten times below the method's error, so a
wrong weight, index or level cannot hide in it.  Lattice stages are checked
at 1e-5 of the largest value of that stage.  Against the exact sum (direct
minus cutoff, the plain definition) the bound is the method's: 4e-4 B(x)."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from oracle import msm
from gpu_util import flat_index

pytestmark = pytest.mark.gpu

CP_DEVICE_ATOMS_OUTSIDE = 0x4


def _domain(atoms):
    a = np.asarray(atoms, dtype=np.float32)
    return tuple(float(v) for v in a[:, :3].min(0)), tuple(float(v) for v in a[:, :3].max(0))


def _run(w, h0, domain=None, out=None, accumulate=False, workspace=None):
    a = torch.from_numpy(w.atoms).cuda()
    dom = domain if domain is not None else _domain(w.atoms)
    V = cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom, out=out, accumulate=accumulate,
                         workspace=workspace)
    torch.cuda.synchronize()
    return V, dom


def _bound(w, pts=None):
    return msm.abs_charge_bound(w.atoms, w.shape, w.origin, w.h, w.cutoff, points=pts)


def _check(got, ref, bound, rel, name):
    err = np.abs(got - ref)
    worst = float((err / bound).max())
    assert np.all(err <= rel * bound), f"{name}: max |dV|/B = {worst:.3e} > {rel:.1e}"


CASES = [
    # name, workload, h0
    ("ragged", workloads.random_case(701, 700, (37, 21, 19), h=0.5, origin=(-1.0, 0.5, 2.0), margin=5.0,
                                     cutoff=4.0, bin_size=2.0), 0.7),
    ("offgrid_domain", workloads.random_case(702, 500, (24, 24, 24), h=0.4, origin=(3.0, -2.0, 0.0),
                                             margin=9.0, cutoff=3.0, bin_size=1.5), 0.5),
    ("coarse", workloads.random_case(703, 900, (30, 30, 30), h=0.5, origin=(0.0, 0.0, 0.0), margin=2.0,
                                     cutoff=5.0, bin_size=2.5), 2.5),
    # the largest stencil the library takes: R = ceil(2c/h0) = 24
    ("max_radius", workloads.random_case(707, 300, (16, 14, 12), h=0.5, origin=(0.0, 0.0, 0.0), margin=2.0,
                                         cutoff=6.0, bin_size=3.0), 0.5),
    # grid spacing above the lattice spacing: the per-quad interpolation kernel
    ("grid_coarser_than_lattice", workloads.random_case(706, 600, (21, 14, 11), h=1.0, origin=(0.5, -1.0, 2.0),
                                                        margin=3.0, cutoff=3.0, bin_size=1.5), 0.7),
    # 5000 A from the coordinate origin with grid points that are not fp32
    # numbers: point lattice coordinates are formed from the grid origin's
    # offset to the lattice origin, so their rounding does not grow with 5000 A
    ("far_origin", workloads.random_case(708, 500, (20, 14, 11), h=0.37,
                                         origin=(5000.1234567, -4999.2345679, 2500.31415), margin=3.0,
                                         cutoff=3.0, bin_size=1.5), 0.7),
    ("far_origin_coarse_grid", workloads.random_case(709, 500, (15, 12, 9), h=1.03,
                                                     origin=(-5000.4321, 3000.777, 4999.9), margin=3.0,
                                                     cutoff=3.0, bin_size=1.5), 0.7),
]


@pytest.mark.parametrize("name,w,h0", CASES, ids=[c[0] for c in CASES])
def test_longrange_matches_oracle_everywhere(name, w, h0):
    V, dom = _run(w, h0)
    got = V.cpu().numpy().reshape(-1).astype(np.float64)
    ref = msm.long_range(w.atoms, w.shape, w.origin, w.h, dom[0], dom[1], w.cutoff, h0)
    _check(got, ref, _bound(w), 1e-5, name)
    assert cp.device_status() == 0


def test_lattice_stages_match_oracle():
    """q on level 0, and every level's potentials e(l), read from the workspace."""
    name, w, h0 = CASES[0]
    a = torch.from_numpy(w.atoms).cuda()
    dom = _domain(w.atoms)
    L = cp.msm_layout(len(w.atoms), w.shape, w.origin, w.h, w.cutoff, h0, dom)
    ws = torch.empty(L.total_bytes, dtype=torch.uint8, device="cuda")
    cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom, workspace=ws)
    torch.cuda.synchronize()
    geo = msm.geometry(w.shape, w.origin, w.h, dom[0], dom[1], w.cutoff, h0)
    assert L.levels == len(geo.levels)
    R = L.radius

    def lattice(off, dims):
        n = int(np.prod(dims))
        return ws[off: off + 4 * n].view(torch.float32).view(*dims[::-1]).cpu().numpy().astype(np.float64)

    qd, plane = tuple(L.q_dims[0]), int(L.q_plane[0])
    pairs = ws[L.off_q[0]: L.off_q[0] + 8 * plane * qd[2]].view(torch.float32).view(qd[2], plane, 2)
    pairs = pairs.cpu().numpy().astype(np.float64)
    q0 = pairs[:, :qd[0] * qd[1], 0].reshape(qd[2], qd[1], qd[0])
    second = pairs[:, :qd[0] * qd[1], 1].reshape(qd[2], qd[1], qd[0])
    assert np.array_equal(second[:, :-1, :], q0[:, 1:, :]) and not second[:, -1, :].any()
    n0 = geo.levels[0].n
    inner = q0[R:R + n0[2], R:R + n0[1], R:R + n0[0]]
    ref_q0 = msm.anterpolate(w.atoms, geo)
    assert np.abs(inner - ref_q0).max() <= 1e-5 * np.abs(ref_q0).max()
    pad = q0.copy()
    pad[R:R + n0[2], R:R + n0[1], R:R + n0[0]] = 0.0
    assert not pad.any(), "charge lattice padding must be zero"
    ref_e = msm.lattice_potentials(w.atoms, geo)
    for l in range(L.levels):
        e = lattice(L.off_e[l], tuple(L.n[l]))
        assert np.abs(e - ref_e[l]).max() <= 1e-5 * np.abs(ref_e[l]).max(), f"level {l}"


def test_single_level_top_only():
    """A domain small enough that level 0 is the top (dense) level."""
    w = workloads.random_case(704, 120, (8, 8, 8), h=0.5, origin=(0.0, 0.0, 0.0), margin=0.0, cutoff=2.0,
                              bin_size=1.0)
    dom = ((0.0, 0.0, 0.0), (4.0, 4.0, 4.0))
    L = cp.msm_layout(len(w.atoms), w.shape, w.origin, w.h, w.cutoff, 1.0, dom)
    assert L.levels == 1
    V, _ = _run(w, 1.0, domain=dom)
    ref = msm.long_range(w.atoms, w.shape, w.origin, w.h, dom[0], dom[1], w.cutoff, 1.0)
    _check(V.cpu().numpy().reshape(-1).astype(np.float64), ref, _bound(w), 1e-5, "top only")


def test_benchmark_geometry_sampled_and_full_map():
    """200^3 map, 100k atoms, c = 12, h0 = 2 (c/h0 = 6, four levels): sampled
    points against the oracle's multilevel sum; the multilevel map (cutoff +
    long range) against the direct sum within the method's error."""
    w = workloads.make("cutoff_uniform")
    h0 = 2.0
    a = torch.from_numpy(w.atoms).cuda()
    dom = cp.atom_bounds(a)
    V = cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom)
    full = cp.msm_map(a, w.shape, w.origin, w.h, w.cutoff, w.bin_size, h0, capacity=0, domain=dom)
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    pts = workloads.sample_points(w.shape, 512, seed=7001)
    idx = flat_index(w.shape, pts)
    bound = _bound(w, pts)
    ref = msm.long_range(w.atoms, w.shape, w.origin, w.h, dom[0], dom[1], w.cutoff, h0, points=pts)
    got = V.cpu().numpy().reshape(-1).astype(np.float64)[idx]
    _check(got, ref, bound, 1e-5, "benchmark long range")
    vd, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h, points=pts)
    vs, _ = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, w.cutoff, points=pts)
    _check(got, vd - vs, bound, 4e-4, "long range vs exact")
    fm = full.cpu().numpy().reshape(-1).astype(np.float64)[idx]
    _check(fm, vd, bound, 4e-4, "multilevel map vs direct sum")
    assert np.all(np.isfinite(V.cpu().numpy()))


def test_accumulate_adds_to_v():
    name, w, h0 = CASES[0]
    base = torch.randn(w.shape[2], w.shape[1], w.shape[0], device="cuda")
    V1, dom = _run(w, h0)
    V2, _ = _run(w, h0, domain=dom, out=base.clone(), accumulate=True)
    assert torch.equal(V2, base + V1)


def test_deterministic():
    name, w, h0 = CASES[1]
    V1, dom = _run(w, h0)
    V2, _ = _run(w, h0, domain=dom)
    assert torch.equal(V1, V2)


def test_atom_outside_domain_is_left_out_and_flagged():
    name, w, h0 = CASES[0]
    dom = _domain(w.atoms)
    far = w.atoms.copy()
    far[5, 0] = dom[1][0] + 50.0  # outside the box given
    a = torch.from_numpy(far).cuda()
    V = cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom)
    torch.cuda.synchronize()
    assert cp.device_status() & CP_DEVICE_ATOMS_OUTSIDE
    keep = np.delete(far, 5, axis=0)
    V_ref = cp.msm_longrange(torch.from_numpy(keep).cuda(), w.shape, w.origin, w.h, w.cutoff, h0, domain=dom)
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    assert torch.equal(V, V_ref)


def test_no_atoms_gives_zero():
    w = workloads.random_case(705, 1, (12, 12, 12), h=0.5, cutoff=3.0, bin_size=1.5)
    empty = torch.zeros((0, 4), dtype=torch.float32, device="cuda")
    V = cp.msm_longrange(empty, w.shape, w.origin, w.h, w.cutoff, 1.0, domain=((0, 0, 0), (5.5, 5.5, 5.5)))
    torch.cuda.synchronize()
    assert not V.any()


def test_atom_bounds_exact():
    w = workloads.make("cutoff_large")
    a = torch.from_numpy(w.atoms).cuda()
    lo, hi = cp.atom_bounds(a)
    assert lo == tuple(float(v) for v in w.atoms[:, :3].min(0))
    assert hi == tuple(float(v) for v in w.atoms[:, :3].max(0))


def test_large_clustered_workload_sampled():
    """400^3 map, 800k atoms (30 % in Gaussian clusters), c = 12, h0 = 4 (four
    levels from 57x58x59 nodes): 256 sampled points against the oracle's
    multilevel sum, within 1e-5 of sum |q|/r (a looser scale than B(x),
    from the C oracle, which is fast at this size)."""
    w = workloads.make("cutoff_large")
    h0 = 4.0
    a = torch.from_numpy(w.atoms).cuda()
    dom = cp.atom_bounds(a)
    V = cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom)
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    pts = workloads.sample_points(w.shape, 256, seed=7002)
    got = V.cpu().numpy().reshape(-1).astype(np.float64)[flat_index(w.shape, pts)]
    ref = msm.long_range(w.atoms, w.shape, w.origin, w.h, dom[0], dom[1], w.cutoff, h0, points=pts)
    _, scale = oracle.direct(w.atoms, w.shape, w.origin, w.h, points=pts)
    _check(got, ref, scale, 1e-5, "large clustered long range")


def test_public_api_with_host_arrays():
    """numpy atoms in, host V out (pinned copies through the library): the
    same maps as with device tensors, for the long-range part and for the
    multilevel map."""
    name, w, h0 = CASES[0]
    dom = _domain(w.atoms)
    host_long = cp.msm_longrange(w.atoms, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom)
    host_map = cp.msm_map(w.atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, h0, capacity=16, domain=dom)
    assert not host_long.is_cuda and not host_map.is_cuda
    a = torch.from_numpy(w.atoms).cuda()
    dev_long = cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0, domain=dom)
    dev_map = cp.msm_map(a, w.shape, w.origin, w.h, w.cutoff, w.bin_size, h0, capacity=16, domain=dom)
    torch.cuda.synchronize()
    assert torch.equal(host_long, dev_long.cpu())
    assert torch.equal(host_map, dev_map.cpu())
    # without a domain the binding asks the library for the atoms' bounding box
    auto = cp.msm_longrange(a, w.shape, w.origin, w.h, w.cutoff, h0)
    torch.cuda.synchronize()
    assert torch.equal(auto, dev_long)


def test_longrange_random_geometries():
    """20 seeded random geometries: grid shape 1..29 per axis, spacing 0.2..1.5 A
    (dyadic or not), origin near or 1000..5000 A from the coordinate origin,
    1..1500 atoms, c = 1.5..5 A, h0 = 0.35..1.6 A (one or more levels, both
    interpolation kernels), against the oracle at every point within 1e-5 B(x).
    Calls the library rejects on the host (a stencil beyond its radius limit)
    are skipped."""
    rng = np.random.default_rng(5)
    for it in range(20):
        shape = tuple(int(v) for v in rng.integers(1, 30, size=3))
        h = float(np.float32(rng.choice([0.5, 0.25, 1.0]) if rng.random() < 0.4 else rng.uniform(0.2, 1.5)))
        shift = rng.uniform(1e3, 5e3, 3) * rng.choice([-1, 1], 3) if rng.random() < 0.3 else np.zeros(3)
        origin = tuple(float(np.float32(v)) for v in rng.uniform(-30, 30, 3) + shift)
        n = int(rng.integers(1, 1500))
        c = float(np.float32(rng.uniform(1.5, 5.0)))
        h0 = float(np.float32(rng.uniform(0.35, 1.6)))
        w = workloads.random_case(30_000 + it, n, shape, h=h, origin=origin, margin=float(rng.uniform(0.0, c + 2.0)))
        a = torch.from_numpy(w.atoms).cuda()
        dom = cp.atom_bounds(a)
        try:
            V = cp.msm_longrange(a, w.shape, w.origin, w.h, c, h0, domain=dom)
        except cp.CpError as e:
            assert e.code == -3, e  # CP_ERR_TOO_LARGE
            continue
        torch.cuda.synchronize()
        assert cp.device_status() == 0
        got = V.cpu().numpy().reshape(-1).astype(np.float64)
        ref = msm.long_range(w.atoms, w.shape, w.origin, w.h, dom[0], dom[1], c, h0)
        B = msm.abs_charge_bound(w.atoms, w.shape, w.origin, w.h, c)
        _check(got, ref, B, 1e-5, f"case {it}: shape {shape} h {h:.4g} origin {origin} c {c:.3g} h0 {h0:.3g}")
