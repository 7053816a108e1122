"""Edge cases of the CUDA path at large or awkward sizes, against the oracle."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from gpu_util import assert_within_bound, flat_index, to_dev

pytestmark = pytest.mark.gpu


def test_direct_many_atoms_small_grid():
    """3 million atoms on a 24^3 grid: every cluster split slices the atom
    array; 512 sampled points by the oracle."""
    rng = np.random.default_rng(81)
    shape, h, origin = (24, 24, 24), 0.5, (0.0, 0.0, 0.0)
    n = 3_000_000
    pos = workloads.off_lattice_uniform(rng, n, (-20.0, -20.0, -20.0), (32.0, 32.0, 32.0), origin, h)
    atoms = np.empty((n, 4), dtype=np.float32)
    atoms[:, :3] = pos
    atoms[:, 3] = rng.uniform(-1, 1, n).astype(np.float32)
    a = to_dev(atoms)
    pts = workloads.sample_points(shape, 512, seed=82)
    ref, bound = oracle.direct(atoms, shape, origin, h, points=pts)
    idx = torch.from_numpy(flat_index(shape, pts)).cuda()
    for split in (0, 1, 16):
        V = cp.direct(a, shape, origin, h, split=split, variant=-1 if split == 0 else 7)
        torch.cuda.synchronize()
        assert_within_bound(V.reshape(-1)[idx].cpu().numpy(), ref, bound, f"split {split}")


@pytest.mark.parametrize("K", [0, 8, 16])
def test_cutoff_crowded_bins(K):
    """400 000 atoms in a 12 A box, about 230 per 1 A bin: long per-bin
    sorts, and every bin run split across many shared-memory stages."""
    rng = np.random.default_rng(83)
    shape, h, origin, c, b = (24, 24, 24), 0.5, (0.0, 0.0, 0.0), 3.0, 1.0
    n = 400_000
    pos = workloads.off_lattice_uniform(rng, n, (0.0, 0.0, 0.0), (12.0, 12.0, 12.0), origin, h)
    atoms = np.empty((n, 4), dtype=np.float32)
    atoms[:, :3] = pos
    atoms[:, 3] = rng.uniform(-1, 1, n).astype(np.float32)
    V = cp.cutoff(to_dev(atoms), shape, origin, h, c, b, capacity=K)
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    pts = workloads.sample_points(shape, 256, seed=84)
    ref, bound = oracle.cutoff_brute(atoms, shape, origin, h, c, points=pts)
    got = V.reshape(-1)[torch.from_numpy(flat_index(shape, pts)).cuda()].cpu().numpy()
    assert_within_bound(got, ref, bound, f"K={K}")


def test_concurrent_streams():
    """Two direct maps and two cutoff maps in flight on two streams at once."""
    w1 = workloads.random_case(85, 4000, (48, 32, 16), margin=2.0)
    w2 = workloads.random_case(86, 3000, (40, 40, 8), h=0.4, origin=(1.0, -2.0, 0.5), margin=2.0)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    a1, a2 = to_dev(w1.atoms), to_dev(w2.atoms)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        d1 = cp.direct(a1, w1.shape, w1.origin, w1.h)
        c1 = cp.cutoff(a1, w1.shape, w1.origin, w1.h, 3.0, 1.0)
    with torch.cuda.stream(s2):
        d2 = cp.direct(a2, w2.shape, w2.origin, w2.h)
        c2 = cp.cutoff(a2, w2.shape, w2.origin, w2.h, 2.5, 1.2)
    torch.cuda.synchronize()
    for w, d, c, cc, bb in ((w1, d1, c1, 3.0, 1.0), (w2, d2, c2, 2.5, 1.2)):
        ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
        assert_within_bound(d.cpu().numpy(), ref, bound, "direct")
        ref, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, cc)
        assert_within_bound(c.cpu().numpy(), ref, bound, "cutoff")


def test_bounded_wait_gives_up_and_reports():
    """A wait on a barrier that nothing arrives at runs out after its limit
    (1 ms here), records CP_DEVICE_WAIT_TIMEOUT and returns; the context stays
    usable and the status word is clean again once read."""
    lib = cp.library()
    assert cp.device_status() == 0
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.cp_probe_wait_timeout(1_000_000, flag.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert flag.item() == 1
    assert cp.device_status() & 0x1  # CP_DEVICE_WAIT_TIMEOUT
    assert cp.device_status() == 0  # read and cleared
    # the context still works
    w = workloads.random_case(77, 50, (8, 8, 4))
    V = cp.direct(torch.from_numpy(w.atoms).cuda(), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    assert torch.isfinite(V).all()
    assert lib.cp_probe_wait_timeout(0, flag.data_ptr(), None) == -1
    assert lib.cp_probe_wait_timeout(3_000_000_000, flag.data_ptr(), None) == -1


def test_maximum_grid():
    """The largest grid the library takes, nx*ny*nz just below 2^31
    (2048 x 1024 x 1023 points, an 8.6 GB V): direct, cutoff and long-range
    maps with a few atoms, checked against the oracle at sampled points that
    include the first and the very last grid point."""
    shape, origin, h = (2048, 1024, 1023), (0.0, 0.0, 0.0), 0.5
    assert shape[0] * shape[1] * shape[2] < 2 ** 31
    rng = np.random.default_rng(4242)
    lo = np.array([0.0, 0.0, 0.0])
    hi = np.array([(shape[0] - 1) * h, (shape[1] - 1) * h, (shape[2] - 1) * h])
    cells = rng.integers(0, (hi / h).astype(int), size=(6, 3))
    pos = (cells + rng.uniform(0.1, 0.9, size=(6, 3))) * h
    atoms = np.concatenate([pos, rng.uniform(-1.0, 1.0, size=(6, 1))], axis=1).astype(np.float32)
    atoms[0, :3] = np.float32([1.3, 1.1, 0.7])      # near the first point
    atoms[1, :3] = (hi - 0.3).astype(np.float32)    # near the last point
    a = to_dev(atoms)
    pts = np.concatenate([workloads.sample_points(shape, 300, seed=4243),
                          np.array([[0, 0, 0], [shape[0] - 1, shape[1] - 1, shape[2] - 1],
                                    [shape[0] - 1, 0, shape[2] - 1]])])
    idx = torch.from_numpy(flat_index(shape, pts)).cuda()
    V = torch.empty((shape[2], shape[1], shape[0]), dtype=torch.float32, device="cuda")
    flat = V.view(-1)

    cp.direct(a, shape, origin, h, out=V)
    got = flat[idx].cpu().numpy()
    ref, bound = oracle.direct(atoms, shape, origin, h, points=pts)
    assert_within_bound(got, ref, bound, "direct, maximum grid")

    c, b = 8.0, 16.0
    cp.cutoff(a, shape, origin, h, c, b, 0, out=V)
    got = flat[idx].cpu().numpy()
    refc, boundc = oracle.cutoff_brute(atoms, shape, origin, h, c, points=pts)
    assert np.all(np.abs(got - refc) <= 2e-4 * boundc + 1e-30)

    from oracle import msm
    dom = cp.atom_bounds(a)
    cp.msm_longrange(a, shape, origin, h, c, 4.0, domain=dom, out=V)
    got = flat[idx].cpu().numpy()
    refl = msm.long_range(atoms, shape, origin, h, dom[0], dom[1], c, 4.0, points=pts)
    bl = msm.abs_charge_bound(atoms, shape, origin, h, c, points=pts)
    assert np.all(np.abs(got - refl) <= 1e-5 * bl)
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    del V, flat
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 37, 1), (2, 1, 9), (3, 3, 3), (1000, 1, 1), (1, 1, 300),
                                   (5, 1, 64)])
def test_degenerate_grids(shape):
    """Grids one or two points wide along some axes: the planner's choice, the
    shared-patch and 2-point shapes with and without a cluster split (rows and
    planes past the grid are computed and not stored), and the cutoff map, each
    against the oracle at every point."""
    w = workloads.random_case(90 + sum(shape), 500, shape, h=0.5, origin=(-1.0, 2.0, 0.5), margin=3.0)
    a = to_dev(w.atoms)
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    V = cp.direct(a, w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    assert_within_bound(V.cpu().numpy(), ref, bound, f"{shape} planner")
    for v in (10, 12, 16, 17, 18):
        for split in (1, 5):
            V = cp.direct(a, w.shape, w.origin, w.h, variant=v, split=split)
            torch.cuda.synchronize()
            assert_within_bound(V.cpu().numpy(), ref, bound, f"{shape} variant {v} split {split}")
    c, b = 2.5, 1.0
    refc, boundc = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    for K in (0, 16):
        Vc = cp.cutoff(a, w.shape, w.origin, w.h, c, b, capacity=K)
        torch.cuda.synchronize()
        assert_within_bound(Vc.cpu().numpy(), refc, boundc, f"{shape} cutoff K={K}")
    assert cp.device_status() == 0


@pytest.mark.parametrize("offset", [0.0, 200.0, 5000.0])
def test_grids_far_from_the_coordinate_origin(offset):
    """Differences are formed as index * h + (origin - atom), rounded once, so the
    accuracy does not depend on where the grid sits: a grid 5000 A from the
    coordinate origin with h = 0.37 A (grid points not exact in fp32) meets the
    same bound at every point.  Forming the point first and subtracting the atom
    after would carry ulp(5000)/2 = 2.4e-4 A into every difference, above the
    bound for atoms 0.1 A from a point."""
    origin = (offset + 0.1234567, -offset + 0.7654321, offset / 2 + 0.31415)
    w = workloads.random_case(95, 1200, (20, 14, 11), h=0.37, origin=origin, margin=2.5)
    a = to_dev(w.atoms)
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    for v, split in ((-1, 0), (7, 1), (18, 3), (10, 1)):
        V = cp.direct(a, w.shape, w.origin, w.h, variant=v, split=split)
        torch.cuda.synchronize()
        assert_within_bound(V.cpu().numpy(), ref, bound, f"offset {offset} variant {v}")
    c, b = 2.0, 0.9
    refc, boundc = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    for K in (0, 16):
        Vc = cp.cutoff(a, w.shape, w.origin, w.h, c, b, capacity=K)
        torch.cuda.synchronize()
        assert_within_bound(Vc.cpu().numpy(), refc, boundc, f"offset {offset} cutoff K={K}")
    assert cp.device_status() == 0


def test_random_geometries():
    """60 seeded random geometries: grid shape 1..39 per axis, spacing 0.2..1.5 A
    (dyadic or not), origin near or 1000..5000 A from the coordinate origin,
    1..2500 atoms, cutoff 1..6 A, bin 0.5..3 A, a random capacity, patch shape and
    cluster split.  Direct (planner and forced) and cutoff maps against the oracle
    at every point, a clean device status after each call.  Calls the library
    rejects on the host (offset lists beyond its limit) are skipped."""
    rng = np.random.default_rng(606)
    for it in range(60):
        shape = tuple(int(v) for v in rng.integers(1, 40, size=3))
        h = float(np.float32(rng.choice([0.5, 0.25, 1.0]) if rng.random() < 0.4 else rng.uniform(0.2, 1.5)))
        shift = rng.uniform(1e3, 5e3, 3) * rng.choice([-1, 1], 3) if rng.random() < 0.3 else np.zeros(3)
        origin = tuple(float(np.float32(v)) for v in rng.uniform(-50, 50, 3) + shift)
        n = int(rng.integers(1, 2500))
        c = float(np.float32(rng.uniform(1.0, 6.0)))
        b = float(np.float32(rng.uniform(0.5, 3.0)))
        w = workloads.random_case(20_000 + it, n, shape, h=h, origin=origin, margin=float(rng.uniform(0.0, c + 2.0)))
        a = to_dev(w.atoms)
        tag = f"case {it}: shape {shape} h {h:.4g} origin {origin} n {n} c {c:.3g} b {b:.3g}"
        ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
        v, s = int(rng.integers(0, len(cp.DIRECT_VARIANTS))), int(rng.choice([1, 2, 3, 4, 6, 8]))
        for kw in ({}, {"variant": v, "split": s}):
            V = cp.direct(a, w.shape, w.origin, w.h, **kw)
            torch.cuda.synchronize()
            assert_within_bound(V.cpu().numpy(), ref, bound, f"{tag} direct {kw}")
            assert cp.device_status() == 0, tag
        K = int(rng.choice([0, 8, 16]))
        try:
            Vc = cp.cutoff(a, w.shape, w.origin, w.h, c, b, capacity=K)
        except cp.CpError as e:
            assert e.code == -3, tag  # CP_ERR_TOO_LARGE: offset list beyond the library's limit
            continue
        torch.cuda.synchronize()
        refc, boundc = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
        assert_within_bound(Vc.cpu().numpy(), refc, boundc, f"{tag} cutoff K={K}")
        assert cp.device_status() == 0, tag
