"""Parity of the comparison kernels (the pages' scatter, gather, coarsened and
coalesced direct sums, and the 27-bin hard-cutoff map) against the fp64
oracle, within |V_gpu - V_ref| <= 2e-4 * sum |q|/r."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from gpu_util import assert_within_bound, flat_index, to_dev

pytestmark = pytest.mark.gpu

STRATEGIES = sorted(cp.DIRECT_STRATEGIES)


@pytest.mark.parametrize("strategy", STRATEGIES)
@pytest.mark.parametrize("seed,n,shape,h,origin", [
    (501, 700, (37, 21, 3), 0.37, (-3.25, 1.5, -2.0)),   # ragged x (not a multiple of 4 or 128)
    (502, 9000, (40, 12, 2), 0.5, (0.0, 0.0, 0.0)),      # three constant-memory chunks
    (503, 1, (5, 3, 2), 0.5, (1.0, 1.0, 1.0)),
])
def test_direct_strategy_small(strategy, seed, n, shape, h, origin):
    w = workloads.random_case(seed, n, shape, h=h, origin=origin, margin=2.0)
    V = cp.direct_variant(strategy, to_dev(w.atoms), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    assert_within_bound(V.cpu().numpy(), ref, bound, f"{strategy} {w.name}")


@pytest.mark.parametrize("strategy", STRATEGIES)
def test_direct_strategy_plane_workload(strategy):
    """The pwwt.cn benchmark's case: z-index 10 plane of 100x100x50, 10 000 atoms."""
    w = workloads.make("direct_plane")
    V = cp.direct_variant(strategy, to_dev(w.atoms), w.shape, w.origin, w.h)
    torch.cuda.synchronize()
    ref, bound = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    assert_within_bound(V.cpu().numpy(), ref, bound, strategy)


@pytest.mark.parametrize("strategy", STRATEGIES)
def test_direct_strategy_zero_atoms(strategy):
    out = torch.full((2, 3, 5), 7.0, device="cuda")
    cp.direct_variant(strategy, torch.zeros((0, 4), dtype=torch.float32, device="cuda"), (5, 3, 2),
                      (0, 0, 0), 0.5, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_direct_strategy_rejects_unknown():
    lib = cp.library()
    a = torch.zeros((4, 4), device="cuda")
    V = torch.zeros(8, device="cuda")
    assert lib.cp_direct_variant(7, a.data_ptr(), 4, *cp._grid((2, 2, 2), (0, 0, 0), 0.5), V.data_ptr(), None) == -1


@pytest.mark.parametrize("seed,n,shape,h,origin,c", [
    (511, 1500, (24, 20, 17), 0.5, (0.0, 0.0, 0.0), 3.0),
    (512, 900, (19, 23, 16), 0.4, (-2.1, 0.7, 3.3), 2.5),
    (513, 500, (16, 16, 1), 0.5, (0.0, 0.0, 5.0), 2.0),
])
def test_cutoff27_small(seed, n, shape, h, origin, c):
    w = workloads.random_case(seed, n, shape, h=h, origin=origin, margin=c + 1.0)
    V = cp.cutoff27(to_dev(w.atoms), w.shape, w.origin, w.h, c)
    torch.cuda.synchronize()
    ref, bound = oracle.cutoff_hard(w.atoms, w.shape, w.origin, w.h, c)
    assert_within_bound(V.cpu().numpy(), ref, bound, w.name)


def test_cutoff27_uniform_workload_sampled():
    w = workloads.make("cutoff_uniform")
    V = cp.cutoff27(to_dev(w.atoms), w.shape, w.origin, w.h, w.cutoff)
    torch.cuda.synchronize()
    pts = workloads.sample_points(w.shape, 2048, seed=4100)
    ref, bound = oracle.cutoff_hard(w.atoms, w.shape, w.origin, w.h, w.cutoff, points=pts)
    got = V.reshape(-1)[torch.from_numpy(flat_index(w.shape, pts)).cuda()].cpu().numpy()
    assert_within_bound(got, ref, bound, w.name)
