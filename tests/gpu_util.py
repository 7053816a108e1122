"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

import oracle

# Accuracy bound: |V_gpu - V_ref| <= REL * sum_{contributing a} |q_a| / r_{a,g}
REL = 2e-4


def assert_within_bound(v_gpu, v_ref, bound, label=""):
    v_gpu = np.asarray(v_gpu, dtype=np.float64).reshape(-1)
    v_ref = np.asarray(v_ref, dtype=np.float64).reshape(-1)
    bound = np.asarray(bound, dtype=np.float64).reshape(-1)
    assert v_gpu.shape == v_ref.shape
    assert np.all(np.isfinite(v_gpu)), f"{label}: non-finite values"
    err = np.abs(v_gpu - v_ref)
    lim = REL * bound
    ratio = np.max(err / np.maximum(lim, 1e-300)) if err.size else 0.0
    bad = err > lim
    assert not bad.any(), (f"{label}: {int(bad.sum())} of {err.size} points beyond {REL} * sum|q|/r "
                           f"(worst ratio {ratio:.3g})")
    return float(ratio)


def flat_index(shape, pts):
    nx, ny, _ = shape
    pts = np.asarray(pts, dtype=np.int64)
    return pts[:, 0] + nx * (pts[:, 1] + ny * pts[:, 2])


def to_dev(atoms):
    return torch.from_numpy(np.ascontiguousarray(atoms)).cuda()
