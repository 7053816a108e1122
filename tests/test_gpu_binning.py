"""Binning on the GPU is bit-exact against the oracle's counting sort:
counts, prefix sums, bin-sorted indices and atoms, fixed-capacity slots
with pads, and the counters."""
import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


def _compare(atoms, shape, origin, h, c, b, K):
    got = cp.bin_atoms(to_dev(atoms), shape, origin, h, c, b, capacity=K)
    torch.cuda.synchronize()
    ref = oracle.bin_atoms(atoms, shape, origin, h, c, b, capacity=K)
    L = got["layout"]
    assert list(L.nb) == list(ref["nb"])
    assert np.array_equal(got["count"].cpu().numpy(), ref["count"])
    assert np.array_equal(got["start"].cpu().numpy(), ref["start"])
    nb_ = ref["n_binned"]
    assert np.array_equal(got["csr_index"][:nb_].cpu().numpy(), ref["csr_index"])
    assert np.array_equal(got["csr_atoms"][:nb_].cpu().numpy().view(np.uint32), ref["csr_atoms"].view(np.uint32))
    assert np.array_equal(got["padded"].cpu().numpy().view(np.uint32), ref["padded"].view(np.uint32))
    st = cp.cutoff_stats(got["workspace"], atoms.shape[0], shape, origin, h, c, b, K)
    assert st["n_binned"] == nb_
    assert st["n_dropped"] == ref["n_dropped"]
    assert st["n_overflow"] == int(np.maximum(ref["count"] - K, 0).sum())
    assert st["max_bin_count"] == int(ref["count"].max(initial=0))
    return st


@pytest.mark.parametrize("K", [0, 8, 16])
@pytest.mark.parametrize("seed,n,shape,h,origin,c,b", [
    (401, 3000, (24, 20, 17), 0.5, (0.0, 0.0, 0.0), 3.0, 1.0),
    (402, 5000, (19, 23, 16), 0.4, (-2.1, 0.7, 3.3), 2.5, 0.6),
    (403, 1, (8, 8, 8), 0.5, (0.0, 0.0, 0.0), 2.0, 1.0),
])
def test_binning_small(K, seed, n, shape, h, origin, c, b):
    w = workloads.random_case(seed, n, shape, h=h, origin=origin, margin=c + 2.0)
    _compare(w.atoms, shape, origin, h, c, b, K)


def test_binning_faces_crowded_and_dropped():
    rng = np.random.default_rng(3)
    shape, h, origin, c, b = (16, 16, 16), 0.5, (0.0, 0.0, 0.0), 2.0, 1.0
    nb, bo, m = oracle.bin_geometry(shape, origin, h, c, b)
    rows = []
    for k in range(40):  # exactly on bin faces
        rows.append([bo[0] + np.float32(k % 9) * np.float32(b), bo[1] + np.float32(3 * b), rng.uniform(0, 7), 0.5])
    for t in range(300):  # one crowded bin
        rows.append([3.2 + 0.001 * t, 2.5, 4.75, (t % 7) - 3.0])
    rows += [[np.nan, 0, 0, 1], [-1e9, 0, 0, 1], [0, 1e9, 0, 1], [np.inf, -np.inf, 0, 1]]
    atoms = np.asarray(rows, dtype=np.float32)
    for K in (0, 8, 16):
        st = _compare(atoms, shape, origin, h, c, b, K)
        assert st["n_dropped"] == 4 and st["max_bin_count"] >= 300


def test_binning_zero_atoms():
    atoms = np.zeros((0, 4), dtype=np.float32)
    _compare(atoms, (8, 8, 8), (0.0, 0.0, 0.0), 0.5, 2.0, 1.0, 16)


@pytest.mark.parametrize("name", ["cutoff_uniform", "cutoff_large"])
def test_binning_workloads(name):
    w = workloads.make(name)
    for K in (0, 8, 16):
        _compare(w.atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, K)
