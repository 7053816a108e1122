"""cp_cutoff_no_alloc: the cutoff map for callers that cannot allocate device
memory (their device memory belongs to another allocator, or they may not
allocate once running).  Its scratch is a fixed 16 MiB array inside the
library, shared by every call on a device.

Checked through the C ABI against the existing entry point cp_cutoff on
calls in a row with different inputs: a small map, then a large one, then
the small one again, so that the last call runs over an array still holding
the bins of a bigger map (anything left over from it would show), within the
accuracy bound the other parity tests use: |dV| <= 2e-4 * sum_{r<c} |q|/r,
and bit for bit.  This file is collected last so that a failure here cannot
hide failures elsewhere."""
import ctypes

import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
import oracle
import workloads
from gpu_util import assert_within_bound, flat_index

pytestmark = pytest.mark.gpu

CP_ERR_TOO_LARGE = -3


def _no_alloc(w, atoms_dev, K=16):
    lib = cp.library()
    V = torch.full((w.shape[2], w.shape[1], w.shape[0]), float("nan"), device="cuda")
    rc = lib.cp_cutoff_no_alloc(atoms_dev.data_ptr(), int(atoms_dev.shape[0]), *cp._grid(w.shape, w.origin, w.h),
                                float(np.float32(w.cutoff)), float(np.float32(w.bin_size)), K, V.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0, cp.status_string(rc)
    return V


def _cases():
    small = workloads.random_case(611, 1500, (24, 20, 17), h=0.5, origin=(-1.0, 0.5, 2.0), margin=4.0,
                                  cutoff=3.0, bin_size=1.0)
    big = workloads.make("cutoff_uniform")  # about 12 MiB of scratch: fits the 16 MiB array
    return [small, big, small]


def test_no_alloc_matches_cutoff_on_calls_in_a_row():
    cases = _cases()
    devs = [torch.from_numpy(w.atoms).cuda() for w in cases]
    # two calls in a row on the shared array, then the existing entry point
    got = [_no_alloc(w, a) for w, a in zip(cases, devs)]
    torch.cuda.synchronize()
    ref = [cp.cutoff(a, w.shape, w.origin, w.h, w.cutoff, w.bin_size, capacity=16) for w, a in zip(cases, devs)]
    torch.cuda.synchronize()
    assert cp.device_status() == 0
    for w, g, r in zip(cases, got, ref):
        g_np = g.cpu().numpy().reshape(-1).astype(np.float64)
        r_np = r.cpu().numpy().reshape(-1).astype(np.float64)
        if w.n_points <= 20000:
            _, bound = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, w.cutoff)
            idx = np.arange(w.n_points)
        else:
            pts = workloads.sample_points(w.shape, 4096, seed=4099)
            _, bound = oracle.cutoff_binned(w.atoms, w.shape, w.origin, w.h, w.cutoff, w.bin_size, points=pts)
            idx = flat_index(w.shape, pts)
            assert np.all(np.isfinite(g_np))
        assert_within_bound(g_np[idx], r_np[idx], bound, w.name)
        # same kernels on the same bins: the results are in fact identical
        assert np.array_equal(g_np, r_np)


def test_no_alloc_rejects_maps_beyond_its_array():
    w = workloads.random_case(612, 10, (400, 400, 400), cutoff=12.0, bin_size=4.0)
    need = cp.cutoff_workspace_bytes(800_000, w.shape, w.origin, w.h, 12.0, 4.0, 16)
    assert need > (16 << 20)
    atoms = torch.zeros((800_000, 4), dtype=torch.float32, device="cuda")
    V = torch.zeros(1, device="cuda")  # never written: the call is refused on the host
    rc = cp.library().cp_cutoff_no_alloc(atoms.data_ptr(), 800_000, *cp._grid(w.shape, w.origin, w.h), 12.0, 4.0,
                                         16, V.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == CP_ERR_TOO_LARGE
    assert V.item() == 0.0
