"""The bounds-checked build (libcpmap_checked.so, -DCP_BOUNDS_CHECKS) on the
GPU.  Every runtime-computed index of the kernels' memory accesses is tested
in that build; a violation sets CP_DEVICE_RANGE and skips the access.  A
child process with CPMAP_CHECKED=1 runs the direct map (every patch shape,
cluster splits 1, 8 and 16, an odd nx), the cutoff map with capacity 0, 8
and 16 (a ragged grid, a crowded bin, the 200^3 benchmark map), the binning
stage and the long-range part (both interpolation kernels, one and four
levels), and a grid 5000 A from the coordinate origin whose points are not
fp32 numbers (the kernels' relative-difference paths); the device status
must stay clean and the maps must equal the release build's bit for bit."""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import direct_coulomb_summation_gb300 as cp
from direct_coulomb_summation_gb300 import build as libbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent('''
    import sys, numpy as np, torch
    sys.path.insert(0, ROOT)
    import direct_coulomb_summation_gb300 as cp
    import workloads

    def runs():
        out = {}
        w = workloads.random_case(901, 1300, (37, 13, 9), h=0.5, origin=(-1.0, 0.5, 2.0), margin=2.0)
        a = torch.from_numpy(w.atoms).cuda()
        for v in sorted(cp.DIRECT_VARIANTS):
            for s in (1, 8, 16):
                out[f"direct_{v}_{s}"] = cp.direct(a, w.shape, w.origin, w.h, variant=v, split=s)
        out["direct_plan"] = cp.direct(a, w.shape, w.origin, w.h)
        c = workloads.random_case(902, 2000, (30, 22, 17), h=0.5, origin=(0.0, 0.0, 0.0), margin=3.0,
                                  cutoff=3.0, bin_size=1.0)
        ac = torch.from_numpy(c.atoms).cuda()
        crowd = c.atoms.copy()
        crowd[:300, :3] = np.float32([5.23, 4.31, 3.77]) + np.float32(0.01) * np.arange(300, dtype=np.float32)[:, None] % 1
        acr = torch.from_numpy(crowd).cuda()
        for K in (0, 8, 16):
            out[f"cutoff_{K}"] = cp.cutoff(ac, c.shape, c.origin, c.h, c.cutoff, c.bin_size, K)
            out[f"crowd_{K}"] = cp.cutoff(acr, c.shape, c.origin, c.h, c.cutoff, c.bin_size, K)
        b = cp.bin_atoms(ac, c.shape, c.origin, c.h, c.cutoff, c.bin_size, 16)
        out["bins_csr"] = b["csr_atoms"].clone()
        out["bins_padded"] = b["padded"].clone()
        big = workloads.make("cutoff_uniform")
        ab = torch.from_numpy(big.atoms).cuda()
        out["cutoff_big"] = cp.cutoff(ab, big.shape, big.origin, big.h, big.cutoff, big.bin_size, 0)
        dom = cp.atom_bounds(ab)
        out["msm_big"] = cp.msm_longrange(ab, big.shape, big.origin, big.h, big.cutoff, 2.0, domain=dom)
        m = workloads.random_case(903, 600, (21, 14, 11), h=1.0, origin=(0.5, -1.0, 2.0), margin=3.0,
                                  cutoff=3.0, bin_size=1.5)
        am = torch.from_numpy(m.atoms).cuda()
        out["msm_quad"] = cp.msm_longrange(am, m.shape, m.origin, m.h, m.cutoff, 0.7, domain=cp.atom_bounds(am))
        t = workloads.random_case(904, 120, (8, 8, 8), h=0.5, cutoff=2.0, bin_size=1.0, margin=0.0)
        at = torch.from_numpy(t.atoms).cuda()
        out["msm_top"] = cp.msm_longrange(at, t.shape, t.origin, t.h, t.cutoff, 1.0,
                                          domain=((0.0, 0.0, 0.0), (4.0, 4.0, 4.0)))
        # grid points that are not fp32 numbers: the kernels' relative differences
        f = workloads.random_case(905, 900, (20, 14, 11), h=0.37, origin=(5000.1234567, -4999.2345679, 2500.31415),
                                  margin=3.0, cutoff=3.0, bin_size=1.5)
        af = torch.from_numpy(f.atoms).cuda()
        for v in (4, 7, 12, 16, 18):
            for s in (1, 8):
                out[f"far_direct_{v}_{s}"] = cp.direct(af, f.shape, f.origin, f.h, variant=v, split=s)
        for K in (0, 16):
            out[f"far_cutoff_{K}"] = cp.cutoff(af, f.shape, f.origin, f.h, f.cutoff, f.bin_size, K)
        out["far_msm"] = cp.msm_longrange(af, f.shape, f.origin, f.h, f.cutoff, 0.7, domain=cp.atom_bounds(af))
        # nx = 20: the last brick's second half-row of the interpolation lies past the grid
        for h0 in (0.4, 0.7, 1.0):
            out[f"far_msm_{h0}"] = cp.msm_longrange(af, f.shape, f.origin, f.h, f.cutoff, h0,
                                                    domain=cp.atom_bounds(af))
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in out.items()}

    res = runs()
    status = cp.device_status()
    np.savez(OUT, status=np.array([status]), lib=np.array([cp._lib.library_path()]), **res)
''')


def test_checked_build_is_clean_and_identical(tmp_path):
    libbuild.build(checked=True)
    out = str(tmp_path / "checked.npz")
    code = SCRIPT.replace("ROOT", repr(ROOT)).replace("OUT", repr(out))
    env = dict(os.environ, CPMAP_CHECKED="1")
    proc = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    got = np.load(out)
    assert str(got["lib"][0]).endswith("libcpmap_checked.so")
    assert int(got["status"][0]) == 0, f"checked build reported device status {int(got['status'][0]):#x}"
    # the same calls through the release library in this process
    env_code = SCRIPT.replace("ROOT", repr(ROOT)).replace("OUT", repr(str(tmp_path / "release.npz")))
    proc = subprocess.run([sys.executable, "-c", env_code], env={k: v for k, v in os.environ.items()
                                                                 if k != "CPMAP_CHECKED"},
                          capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    ref = np.load(str(tmp_path / "release.npz"))
    assert str(ref["lib"][0]).endswith("libcpmap.so")
    assert int(ref["status"][0]) == 0
    for key in ref.files:
        if key in ("status", "lib"):
            continue
        assert np.array_equal(got[key], ref[key], equal_nan=True), key
