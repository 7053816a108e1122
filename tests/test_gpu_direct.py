"""GPU parity of the direct sum: the sm_103a kernel (through the C ABI)
against the fp64 oracle, element by element, within
|V_gpu - V_ref| <= 2e-4 * sum_a |q_a| / r  at every checked point."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from gpu_util import assert_within_bound, flat_index, to_dev

pytestmark = pytest.mark.gpu


def _check_full(w, **kw):
    V = cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h, **kw)
    torch.cuda.synchronize()
    assert V.shape == (w.shape[2], w.shape[1], w.shape[0])
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    return assert_within_bound(V.cpu().numpy(), ref, bound, w.name)


@pytest.mark.parametrize("seed,n,shape,h,origin", [
    (101, 1100, (37, 21, 9), 0.37, (-3.25, 1.5, -2.0)),    # 3 atom tiles, ragged x, odd y and z
    (102, 513, (40, 12, 4), 0.5, (0.0, 0.0, 0.0)),          # one atom past a tile
    (103, 64, (5, 3, 2), 0.5, (1.0, 1.0, 1.0)),             # tiny grid
    (104, 2000, (128, 8, 3), 0.25, (-8.0, 0.0, 0.0)),
    (105, 1, (16, 16, 16), 0.5, (0.0, 0.0, 0.0)),           # single atom
    (106, 3000, (100, 100, 1), 0.5, (0.0, 0.0, 5.0)),       # plane
])
def test_direct_small_full_grid(seed, n, shape, h, origin):
    w = workloads.random_case(seed, n, shape, h=h, origin=origin, margin=2.0)
    _check_full(w)


@pytest.mark.parametrize("variant", sorted(cp.DIRECT_VARIANTS))
@pytest.mark.parametrize("split", [1, 2, 3, 5, 8, 11, 15, 16])
def test_direct_every_variant_and_split(variant, split):
    w = workloads.random_case(200 + variant, 1537, (44, 13, 6), h=0.5, origin=(-1.0, 0.0, 2.0), margin=1.0)
    _check_full(w, variant=variant, split=split)


@pytest.mark.parametrize("kind,bound", [("sfu", 1e-6), ("fma", 5e-6)])
def test_rsqrt_routes_error_bound(kind, bound):
    """Both rsqrt routes of the kernels against fp64 1/sqrt over 12 decades."""
    rng = np.random.default_rng(17)
    x = np.exp(rng.uniform(np.log(1e-4), np.log(1e8), 1 << 20)).astype(np.float32)
    x = np.concatenate([x, (2.0 ** np.arange(-40, 40)).astype(np.float32)])
    y = cp.eval_rsqrt(torch.from_numpy(x).cuda(), kind).cpu().numpy().astype(np.float64)
    rel = np.abs(y * np.sqrt(x.astype(np.float64)) - 1.0)
    assert rel.max() <= bound, rel.max()


def test_direct_zero_atoms():
    w = workloads.random_case(1, 0, (12, 5, 3))
    V = cp.direct(torch.zeros((0, 4), dtype=torch.float32, device="cuda"), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    assert torch.count_nonzero(V).item() == 0


def test_direct_unaligned_output_and_odd_nx():
    w = workloads.random_case(7, 700, (13, 7, 5), h=0.5, margin=1.0)
    buf = torch.full((13 * 7 * 5 + 1,), float("nan"), device="cuda")
    out = buf[1:]  # 4-byte aligned only: scalar stores
    cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h, out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[0]).item()
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    assert_within_bound(out.cpu().numpy(), ref, bound)


@pytest.mark.parametrize("variant", sorted(cp.DIRECT_VARIANTS))
@pytest.mark.parametrize("shape,offset", [((13, 7, 5), 1), ((18, 5, 4), 2)])
def test_direct_every_variant_store_paths(variant, shape, offset):
    """Odd nx into a 4-byte aligned output (scalar stores for every shape), and
    nx = 18 into an 8-byte aligned output (float2 stores for the 2-point shapes,
    scalar ones for the 4-point shapes), without and with a 16-CTA split; the
    floats around the output stay untouched."""
    n = shape[0] * shape[1] * shape[2]
    w = workloads.random_case(400 + variant, 700, shape, h=0.5, margin=1.0)
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    for split in (1, 16):
        buf = torch.full((n + offset + 1,), float("nan"), device="cuda")
        out = buf[offset:offset + n]
        cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h, out=out, variant=variant, split=split)
        torch.cuda.synchronize()
        assert torch.isnan(buf[:offset]).all().item() and torch.isnan(buf[-1]).item()
        assert_within_bound(out.cpu().numpy(), ref, bound, f"variant {variant} split {split}")


def test_direct_overwrites_output():
    w = workloads.random_case(8, 300, (16, 8, 4), margin=1.0)
    out = torch.full((4, 8, 16), 1e30, device="cuda")
    cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h, out=out)
    torch.cuda.synchronize()
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    assert_within_bound(out.cpu().numpy(), ref, bound)


def test_direct_deterministic_and_status_clean():
    w = workloads.random_case(9, 5000, (64, 32, 8), margin=2.0)
    a = to_dev(w.atoms)
    v1 = cp.direct(a, w.shape, w.origin, w.h).clone()
    v2 = cp.direct(a, w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    assert torch.equal(v1, v2)
    assert cp.device_status() == 0


def test_direct_host_buffers_match_device():
    w = workloads.random_case(10, 900, (20, 12, 6), margin=1.0)
    v_host = cp.direct(w.atoms, w.shape, w.origin, w.h)  # numpy in, CPU tensor out
    v_dev = cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    assert not v_host.is_cuda
    assert torch.equal(v_host, v_dev.cpu())


def test_direct_plane_workload_full():
    """10 000 atoms, the 100x100 plane z-index 10 of a 100x100x50 grid: every point."""
    w = workloads.make("direct_plane")
    _check_full(w)


@pytest.mark.parametrize("name", ["direct_3d", "direct_protein"])
def test_direct_workload_sampled(name):
    """Full-size grid in the launch configuration the benchmark uses; the
    oracle checks 4096 seeded points."""
    w = workloads.make(name)
    V = cp.direct(to_dev(w.atoms), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    pts = workloads.sample_points(w.shape, 4096, seed=4096)
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h, points=pts)
    got = V.reshape(-1)[torch.from_numpy(flat_index(w.shape, pts)).cuda()].cpu().numpy()
    assert_within_bound(got, ref, bound, name)
    assert cp.device_status() == 0


def test_direct_superposition_on_gpu():
    """V(A u B) = V(A) + V(B) and V(-q) = -V(q) hold for the GPU map too (within fp32)."""
    w = workloads.random_case(11, 2048, (32, 16, 8), margin=1.0)
    a = to_dev(w.atoms)
    vab = cp.direct(a, w.shape, w.origin, w.h).double()
    va = cp.direct(a[:1000].contiguous(), w.shape, w.origin, w.h).double()
    vb = cp.direct(a[1000:].contiguous(), w.shape, w.origin, w.h).double()
    neg = a.clone()
    neg[:, 3] = -neg[:, 3]
    vn = cp.direct(neg, w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    _, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    bound = torch.from_numpy(bound).cuda().reshape(vab.shape)
    assert torch.all((vab - va - vb).abs() <= 2e-4 * bound)
    assert torch.equal(vn, -vab.float())  # exact: each term negates


def test_direct_far_atoms():
    """Atoms 1e17 A away (padding a caller might use; the documented limit is
    1e18 A, where r^2 still fits fp32) contribute nothing measurable, on both
    rsqrt routes and with grid points that are or are not fp32 numbers."""
    pad = np.array([[1e17, 0, 0, 1.0], [0, -1e17, 5, -0.5], [3e16, 2e16, -5e16, 0.7]], dtype=np.float32)
    for h, origin in ((0.5, (0.0, 0.0, 0.0)), (0.37, (1.2345, -0.5432, 2.111))):
        w = workloads.random_case(12, 900, (24, 16, 8), h=h, origin=origin, margin=1.0)
        atoms = np.concatenate([w.atoms, pad])
        ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
        for v in (-1, 7, 17, 18):
            V = cp.direct(to_dev(atoms), w.shape, w.origin, w.h, variant=v)
            torch.cuda.synchronize()
            assert_within_bound(V.cpu().numpy(), ref, bound, f"h {h} variant {v}")
