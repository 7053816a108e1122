"""Pins for the fp64 oracle: closed forms, invariants, library special cases
and an independent route, chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign, a transposed operand, a wrong coefficient, a
non-strict cutoff, a wrong bin rule) fails at least one of them.  The
mutation tests at the end of this file plant such slips in a copy of the
oracle and check that these pins catch every one.

Sources of the pinned facts:
  * V(g) = sum_a q_a / r_{a,g}: PMPP ch.18 notes ("Case study -- electrostatic
    potential map"), section 18.1; pwwt.cn chapter-18 article, section 一.
  * The cutoff term q*(1/r - (GC0 + r^2 (GC1 + r^2 GC2))) for r^2 < c^2: Input
    Binning lecture, slide "Large Bin Cut-off Kernel Code" (24); its
    coefficients are fixed by g(c) = 1/c, g'(c) = -1/c^2, g''(c) = 2/c^3.
  * Bins by dividing a position by the bin size: PMPP ch.18 notes section
    18.5; Input Binning lecture slide "Pseudo Code of an Implementation" (28).
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
from scipy.spatial.distance import cdist

import oracle
import workloads

SQRT3 = math.sqrt(3.0)


def _atoms(rows):
    return np.asarray(rows, dtype=np.float32).reshape(-1, 4)


def _coords(shape, origin, h, points=None):
    pts = workloads.grid_points(shape) if points is None else np.asarray(points)
    o = np.asarray(origin, dtype=np.float32).astype(np.float64)
    return o[None, :] + pts.astype(np.float64) * float(np.float32(h))


# --------------------------------------------------------------------------
# direct sum


def pin_direct_single_charge():
    # grid point (0,0,0) at the origin, one charge at (1/4,1/4,1/4): r = sqrt(3)/4
    a = _atoms([0.25, 0.25, 0.25, 1.5])
    V, B = oracle.direct(a, (3, 1, 1), (0.0, 0.0, 0.0), 0.5)
    # points at x = 0, 0.5, 1.0: dx = 0.25, 0.25, 0.75 with dy = dz = 0.25
    expect = [1.5 / (SQRT3 / 4.0), 1.5 / (SQRT3 / 4.0), 1.5 / math.sqrt(0.75**2 + 2 * 0.0625)]
    assert np.allclose(V, expect, rtol=1e-15, atol=0)
    assert np.allclose(B, np.abs(expect), rtol=1e-15, atol=0)


def pin_direct_shells():
    # six charges at distance d on the axes and eight on the cube corners
    # around grid point (2, 1, 3) of a grid with origin (-1, 2, 0.5), h = 0.5
    h, origin = 0.5, (-1.0, 2.0, 0.5)
    g = np.array([-1.0 + 2 * h, 2.0 + 1 * h, 0.5 + 3 * h])
    d, s = 0.375, 0.625
    rows = []
    for ax in range(3):
        for sign in (-1, 1):
            p = g.copy()
            p[ax] += sign * d
            rows.append([*p, 0.75])
    for sx in (-1, 1):
        for sy in (-1, 1):
            for sz in (-1, 1):
                rows.append([g[0] + sx * s, g[1] + sy * s, g[2] + sz * s, -0.25])
    V, _ = oracle.direct(_atoms(rows), (4, 3, 5), origin, h, points=[[2, 1, 3]])
    expect = 6 * 0.75 / d + 8 * (-0.25) / (s * SQRT3)
    assert abs(V[0] - expect) <= 1e-14 * abs(expect)


def pin_direct_dipole_axis():
    # +q and -q at z = +-s about the origin; points on the z axis at z = D
    q, s = 0.5, 0.25
    a = _atoms([[0.0, 0.0, s, q], [0.0, 0.0, -s, -q]])
    h = 0.5
    V, _ = oracle.direct(a, (1, 1, 6), (0.0, 0.0, 1.0), h)
    D = 1.0 + h * np.arange(6)
    expect = 2 * q * s / (D**2 - s**2)
    assert np.allclose(V, expect, rtol=1e-13, atol=0)


def pin_direct_cdist():
    # the sum is a matrix-vector product with the inverse distance matrix
    w = workloads.random_case(11, 157, (7, 5, 4), h=0.5, origin=(-1.25, 0.5, 2.0), margin=3.0)
    V, B = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    R = cdist(_coords(w.shape, w.origin, w.h), w.atoms[:, :3].astype(np.float64))
    q = w.atoms[:, 3].astype(np.float64)
    assert np.allclose(V, (q[None, :] / R).sum(axis=1), rtol=1e-12, atol=1e-12)
    assert np.allclose(B, (np.abs(q)[None, :] / R).sum(axis=1), rtol=1e-12, atol=0)


def pin_direct_linearity():
    w = workloads.random_case(12, 300, (6, 6, 3), margin=2.0)
    A, Bq = w.atoms[:120], w.atoms[120:]
    vA, _ = oracle.direct(A, w.shape, w.origin, w.h)
    vB, _ = oracle.direct(Bq, w.shape, w.origin, w.h)
    vAB, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    assert np.allclose(vAB, vA + vB, rtol=1e-12, atol=1e-12)
    neg = w.atoms.copy()
    neg[:, 3] = -neg[:, 3]
    vn, _ = oracle.direct(neg, w.shape, w.origin, w.h)
    assert np.array_equal(vn, -vAB)  # negation is exact term by term
    dbl = w.atoms.copy()
    dbl[:, 3] *= 2
    vd, _ = oracle.direct(dbl, w.shape, w.origin, w.h)
    assert np.array_equal(vd, 2 * vAB)  # doubling is exact term by term


def pin_direct_translation():
    # shift atoms and origin by the same lattice vector: V unchanged
    w = workloads.random_case(13, 200, (5, 4, 6), margin=1.0)
    # coordinates on a 2^-10 A raster so that the shifted fp32 values are exact
    w.atoms[:, :3] = np.round(w.atoms[:, :3] * 1024.0) / 1024.0
    shift = np.array([3 * w.h, -2 * w.h, 5 * w.h], dtype=np.float32)
    moved = w.atoms.copy()
    moved[:, :3] += shift
    o2 = tuple(np.asarray(w.origin, dtype=np.float32) + shift)
    v0, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    v1, _ = oracle.direct(moved, w.shape, o2, w.h)
    assert np.allclose(v0, v1, rtol=1e-12, atol=1e-12)


def pin_direct_point_order():
    # a point list gives the same values as the full grid at those points,
    # and the flat layout is x fastest
    w = workloads.random_case(14, 50, (5, 4, 3), margin=1.0)
    full, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    pts = np.array([[4, 0, 0], [0, 3, 0], [1, 2, 2], [4, 3, 2]], dtype=np.int32)
    some, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h, points=pts)
    flat = pts[:, 0] + 5 * (pts[:, 1] + 4 * pts[:, 2])
    assert np.array_equal(full[flat], some)
    # point (4,0,0) is 2 A along x from the origin: check one atom's term directly
    one = w.atoms[:1]
    v, _ = oracle.direct(one, w.shape, w.origin, w.h, points=pts[:1])
    r = np.linalg.norm(np.array([w.origin[0] + 4 * w.h, w.origin[1], w.origin[2]]) - one[0, :3].astype(np.float64))
    assert abs(v[0] - float(one[0, 3]) / r) <= 1e-14 * abs(v[0])


# --------------------------------------------------------------------------
# switched cutoff term


def pin_switch_closed_forms():
    for c in (12.0, 2.5, 7.0):
        # g(c) = 1/c: the term vanishes at the cutoff
        assert abs(oracle.switch_g(c * c, c) - 1.0 / c) <= 1e-15 / c
        assert abs(oracle.switched_term(c * c, c)) <= 1e-15 / c
        # slope and curvature of g match those of 1/r at r = c (central differences)
        e = 1e-3 * c
        g = lambda r: oracle.switch_g(r * r, c)
        d1 = (g(c + e) - g(c - e)) / (2 * e)
        d2 = (g(c + e) - 2 * g(c) + g(c - e)) / (e * e)
        assert abs(d1 - (-1.0 / c**2)) <= 1e-5 / c**2  # truncation 1.5e-6/c^2
        assert abs(d2 - (2.0 / c**3)) <= 1e-4 / c**3
        # so the term itself is flat to second order at c: with f = 1/r - g,
        # f'''(c) = -6/c^4 - 9/c^4, hence f(c - e) ~ (15/6) e^3 / c^4
        t = oracle.switched_term((c - e) ** 2, c)
        assert abs(t - 2.5 * e**3 / c**4) <= 1e-2 * 2.5 * e**3 / c**4
        # at r -> 0 the polynomial tends to 15/(8c)
        assert abs(oracle.switch_g(0.0, c) - 15.0 / (8.0 * c)) <= 1e-15
    # a value in between: c = 2, r = 1 -> g = (1/2)(15/8 - 5/16 + 3/128) = 203/256
    assert abs(oracle.switch_g(1.0, 2.0) - 203.0 / 256.0) <= 1e-15
    assert abs(oracle.switched_term(1.0, 2.0) - (1.0 - 203.0 / 256.0)) <= 1e-15


def pin_cutoff_single_charge():
    # charge at (0.25, 0.25, 0.25); points along x; c = 1.0
    a = _atoms([0.25, 0.25, 0.25, -2.0])
    V, B = oracle.cutoff_brute(a, (4, 1, 1), (0.0, 0.0, 0.0), 0.5, 1.0)
    r2 = np.array([3 * 0.0625, 3 * 0.0625, 0.5625 + 0.125, 1.5625 + 0.125])  # last: r^2 = 1.6875 > 1
    inside = r2 < 1.0
    c = 1.0
    s = r2 / (c * c)
    g = (1 / c) * (15 / 8 - 5 / 4 * s + 3 / 8 * s * s)
    expect = np.where(inside, -2.0 * (1 / np.sqrt(r2) - g), 0.0)
    assert np.allclose(V, expect, rtol=1e-14, atol=1e-15)
    assert np.allclose(B, np.where(inside, 2.0 / np.sqrt(r2), 0.0), rtol=1e-14, atol=0)


def pin_cutoff_strict_boundary():
    # an atom exactly at r = c (3-4-5 triangle, all fp32-exact): excluded
    a = _atoms([[1.5, 2.0, 0.0, 1.0], [0.75, 1.0, 0.0, 1.0]])
    pairs = oracle.pairs_brute(a, (1, 1, 1), (0.0, 0.0, 0.0), 0.5, 2.5)
    assert pairs.tolist() == [[0, 1]]
    V, B = oracle.cutoff_brute(a, (1, 1, 1), (0.0, 0.0, 0.0), 0.5, 2.5)
    assert abs(B[0] - 1.0 / 1.25) <= 1e-15


def pin_cutoff_cdist():
    w = workloads.random_case(21, 240, (6, 5, 5), h=0.5, origin=(0.5, -1.0, 0.0), margin=2.5)
    c = 1.75
    V, B = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    R = cdist(_coords(w.shape, w.origin, w.h), w.atoms[:, :3].astype(np.float64))
    q = w.atoms[:, 3].astype(np.float64)
    inside = R * R < c * c
    s = (R * R) / (c * c)
    term = np.where(inside, 1.0 / R - (1 / c) * (15 / 8 - 5 / 4 * s + 3 / 8 * s * s), 0.0)
    assert inside.sum() > 100
    assert np.allclose(V, term @ q, rtol=1e-11, atol=1e-12)
    assert np.allclose(B, np.where(inside, 1.0 / R, 0.0) @ np.abs(q), rtol=1e-11, atol=0)


def pin_cutoff_large_c_limit():
    # with every pair inside, cutoff + (15/(8c)) sum q  ->  direct, to O(r^2/c^3)
    w = workloads.random_case(22, 150, (5, 5, 4), margin=2.0)
    c = 1.0e4
    vc, _ = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, c)
    vd, Bd = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    qsum = float(w.atoms[:, 3].astype(np.float64).sum())
    rmax = 10.0
    bound = (5 / 4) * rmax**2 / c**3 * np.abs(w.atoms[:, 3]).sum() + 1e-12 * Bd
    assert np.all(np.abs(vc + 15.0 / (8.0 * c) * qsum - vd) <= bound)


def pin_hard_cutoff():
    # closed forms: a single charge at r = sqrt(3)/4 inside c = 0.5, one at r > c outside
    a = _atoms([[0.25, 0.25, 0.25, 1.5], [2.0, 0.0, 0.0, -1.0]])
    V, B = oracle.cutoff_hard(a, (1, 1, 1), (0.0, 0.0, 0.0), 0.5, 0.5)
    assert abs(V[0] - 1.5 / (SQRT3 / 4.0)) <= 1e-14 and abs(B[0] - 1.5 / (SQRT3 / 4.0)) <= 1e-14
    # an atom exactly at r = c is excluded (strict), as in the switched sum
    a2 = _atoms([[1.5, 2.0, 0.0, 1.0], [0.75, 1.0, 0.0, 1.0]])
    V2, _ = oracle.cutoff_hard(a2, (1, 1, 1), (0.0, 0.0, 0.0), 0.5, 2.5)
    assert abs(V2[0] - 1.0 / 1.25) <= 1e-15
    # with every pair inside, the hard-cutoff sum is the direct sum (same terms, same order)
    w = workloads.random_case(23, 130, (5, 4, 3), margin=1.5)
    vh, _ = oracle.cutoff_hard(w.atoms, w.shape, w.origin, w.h, 1.0e4)
    vd, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    assert np.array_equal(vh, vd)
    # cdist special case with a finite cutoff
    c = 1.6
    vh, bh = oracle.cutoff_hard(w.atoms, w.shape, w.origin, w.h, c)
    R = cdist(_coords(w.shape, w.origin, w.h), w.atoms[:, :3].astype(np.float64))
    inside = R * R < c * c
    q = w.atoms[:, 3].astype(np.float64)
    assert inside.sum() > 50
    assert np.allclose(vh, np.where(inside, 1.0 / R, 0.0) @ q, rtol=1e-12, atol=1e-12)
    assert np.allclose(bh, np.where(inside, 1.0 / R, 0.0) @ np.abs(q), rtol=1e-12, atol=0)


# --------------------------------------------------------------------------
# binning and the binned route


def _face_case(seed=31):
    """Tiny case with atoms on bin faces, near r = c of grid points, outside the grid."""
    rng = np.random.default_rng(seed)
    shape, h, origin, c, b = (9, 7, 6), 0.5, (-0.5, 0.25, 1.0), 1.75, 0.75
    w = workloads.random_case(seed, 120, shape, h=h, origin=origin, margin=2.5, cutoff=c, bin_size=b)
    nb, bo, m = oracle.bin_geometry(shape, origin, h, c, b)
    rows = [list(r) for r in w.atoms]
    # on bin faces: x = bo + k*b exactly
    for k in range(3, 9):
        rows.append([float(bo[0] + np.float32(k * b)), float(rng.uniform(0, 3)), float(rng.uniform(1, 3)), 0.5])
        rows.append([float(rng.uniform(-0.5, 3)), float(bo[1] + np.float32(k * b)), float(bo[2] + np.float32(k * b)), -0.5])
    # at r = c exactly from grid points (scaled 3-4-5 triangle: c = 1.75 = 5*0.35 -> not fp32-exact;
    # use offsets whose squares sum to c^2 exactly in double: (1.05, 1.4, 0) -> 1.1025+1.96 = 3.0625)
    g = np.array([origin[0] + 4 * h, origin[1] + 3 * h, origin[2] + 2 * h])
    rows.append([float(np.float32(g[0] + 1.05)), float(np.float32(g[1] + 1.4)), float(g[2]), 1.0])
    rows.append([float(g[0] - 1.75), float(g[1]), float(g[2] + 0.0), -1.0])  # exactly c along -x
    # a crowded bin (more atoms than the capacity used below)
    for t in range(9):
        rows.append([float(bo[0] + np.float32(5.2 * b) + 0.05 * t), float(bo[1] + np.float32(4.3 * b)),
                     float(bo[2] + np.float32(4.6 * b) - 0.04 * t), 0.125 * (t - 4)])
    # far outside the bin grid (dropped)
    rows.append([1e4, 0.0, 0.0, 1.0])
    rows.append([float("-inf"), 0.0, 0.0, 1.0])
    return _atoms(rows), shape, origin, h, c, b


def pin_bin_rule_numpy():
    atoms, shape, origin, h, c, b = _face_case()
    res = oracle.bin_atoms(atoms, shape, origin, h, c, b, capacity=4)
    nb, bo = res["nb"], res["bo"]
    # the geometry, from its definition
    m = math.ceil(c / b)
    assert res["m"] == m
    for d in range(3):
        assert bo[d] == np.float32(np.float64(np.float32(origin[d])) - m * np.float64(np.float32(b)))
        span = (shape[d] - 1) * np.float64(np.float32(h)) + 2 * m * np.float64(np.float32(b))
        assert nb[d] == math.ceil(span / np.float64(np.float32(b))) + 1
    # every atom's bin, re-derived with numpy float32 arithmetic
    with np.errstate(invalid="ignore", over="ignore"):
        u = np.floor((atoms[:, :3] - bo[None, :]) / np.float32(b)).astype(np.float64)
    ok = np.isfinite(u).all(axis=1) & (u >= 0).all(axis=1) & (u < nb[None, :].astype(np.float64)).all(axis=1)
    ui = np.where(ok[:, None], u, 0).astype(np.int64)
    lin = np.where(ok, (ui[:, 2] * nb[1] + ui[:, 1]) * nb[0] + ui[:, 0], -1)
    assert np.array_equal(res["bin_of_atom"], lin)
    nbins = int(np.prod(nb))
    assert np.array_equal(res["count"], np.bincount(lin[ok], minlength=nbins))
    assert res["n_dropped"] == int((~ok).sum()) >= 2
    assert np.array_equal(res["start"], np.concatenate([[0], np.cumsum(res["count"])]))
    # CSR = stable sort by bin (library routine), i.e. ascending index within a bin
    order = np.argsort(np.where(ok, lin, nbins + 1), kind="stable")[: ok.sum()]
    assert np.array_equal(res["csr_index"], order)
    assert np.array_equal(res["csr_atoms"], atoms[order])
    # fixed-capacity slots: first K of each bin, then the pad record
    K = 4
    padded = res["padded"]
    for bi in np.nonzero(res["count"])[0][:200]:
        seg = order[res["start"][bi]: res["start"][bi + 1]]
        n = min(len(seg), K)
        assert np.array_equal(padded[bi, :n], atoms[seg[:n]])
        assert np.all(padded[bi, n:, :3] == oracle.PAD_COORD) and np.all(padded[bi, n:, 3] == 0)
    empty = np.nonzero(res["count"] == 0)[0]
    assert np.all(padded[empty, :, :3] == oracle.PAD_COORD)
    # some bin must overflow K in this case for the check to mean anything
    assert (res["count"] > K).any()


def pin_binned_equals_brute():
    atoms, shape, origin, h, c, b = _face_case()
    pb = oracle.pairs_brute(atoms, shape, origin, h, c)
    pn = oracle.pairs_binned(atoms, shape, origin, h, c, b)
    assert len(pb) > 500
    assert np.array_equal(pb, pn)
    vb, Bb = oracle.cutoff_brute(atoms, shape, origin, h, c)
    vn, Bn = oracle.cutoff_binned(atoms, shape, origin, h, c, b)
    assert np.array_equal(vb, vn)  # same pairs, same order, same fp64 ops
    assert np.array_equal(Bb, Bn)


def pin_binned_equals_brute_random():
    for seed, (shape, h, origin, c, b) in enumerate(
        [((12, 10, 9), 0.5, (0.0, 0.0, 0.0), 2.0, 1.0),
         ((16, 16, 16), 0.25, (-2.0, 1.0, 0.5), 1.5, 0.5),
         ((7, 11, 5), 0.6, (3.0, -4.0, 1.2), 2.2, 1.3)]):
        w = workloads.random_case(40 + seed, 200, shape, h=h, origin=origin, margin=c + 1.0)
        pb = oracle.pairs_brute(w.atoms, w.shape, w.origin, w.h, c)
        pn = oracle.pairs_binned(w.atoms, w.shape, w.origin, w.h, c, b)
        assert np.array_equal(pb, pn)


PINS = {
    "direct": [pin_direct_single_charge, pin_direct_shells, pin_direct_dipole_axis, pin_direct_cdist,
               pin_direct_linearity, pin_direct_translation, pin_direct_point_order],
    "switch": [pin_switch_closed_forms, pin_cutoff_single_charge, pin_cutoff_strict_boundary,
               pin_cutoff_cdist, pin_cutoff_large_c_limit],
    "hard": [pin_hard_cutoff],
    "bins": [pin_bin_rule_numpy, pin_binned_equals_brute, pin_binned_equals_brute_random],
}
ALL_PINS = [p for group in PINS.values() for p in group]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


# --------------------------------------------------------------------------
# mutation tests: each planted slip must make at least one pin fail

MUTANTS = [
    ("direct_drop_last_atom", "for (long a = 0; a < c->n_atoms; ++a) {\n            const float *at = c->atoms + 4 * a;\n            double dx = x - (double)at[0];\n            double dy = y - (double)at[1];\n            double dz = z - (double)at[2];\n            double r = sqrt",
     "for (long a = 0; a + 1 < c->n_atoms; ++a) {\n            const float *at = c->atoms + 4 * a;\n            double dx = x - (double)at[0];\n            double dy = y - (double)at[1];\n            double dz = z - (double)at[2];\n            double r = sqrt", "direct"),
    ("direct_sign_dx", "double dx = x - (double)at[0];\n            double dy = y - (double)at[1];\n            double dz = z - (double)at[2];\n            double r = sqrt",
     "double dx = x + (double)at[0];\n            double dy = y - (double)at[1];\n            double dz = z - (double)at[2];\n            double r = sqrt", "direct"),
    ("direct_transposed_yz", "double dy = y - (double)at[1];\n            double dz = z - (double)at[2];\n            double r = sqrt",
     "double dy = y - (double)at[2];\n            double dz = z - (double)at[1];\n            double r = sqrt", "direct"),
    ("point_index_j_for_k", "*z = g->oz + (double)k * g->h;", "*z = g->oz + (double)j * g->h;", "direct"),
    ("bound_signed_q", "b += fabs(q) / r;", "b += q / r;", "direct"),
    ("hard_not_strict", "            double r2 = dx * dx + dy * dy + dz * dz;\n            if (r2 < c2) {\n                double q = (double)at[3];\n                double r = sqrt(r2);",
     "            double r2 = dx * dx + dy * dy + dz * dz;\n            if (r2 <= c2) {\n                double q = (double)at[3];\n                double r = sqrt(r2);", "hard"),
    ("hard_bound_signed", "                v += q / r;\n                b += fabs(q) / r;\n            }\n        }\n        c->V[p] = v;\n        if (c->B) c->B[p] = b;\n    }\n}\n\nint or_cutoff_hard",
     "                v += q / r;\n                b += q / r;\n            }\n        }\n        c->V[p] = v;\n        if (c->B) c->B[p] = b;\n    }\n}\n\nint or_cutoff_hard", "hard"),
    ("switch_coef_gc1", "(5.0 / 4.0) * s", "(5.0 / 8.0) * s", "switch"),
    ("switch_coef_gc2", "(3.0 / 8.0) * s * s", "(3.0 / 4.0) * s * s", "switch"),
    ("switch_sign", "return 1.0 / sqrt(r2) - or_switch_g(r2, c);", "return 1.0 / sqrt(r2) + or_switch_g(r2, c);", "switch"),
    ("cutoff_not_strict", "            double r2 = dx * dx + dy * dy + dz * dz;\n            if (r2 < c2) {\n                double q",
     "            double r2 = dx * dx + dy * dy + dz * dz;\n            if (r2 <= c2) {\n                double q", "switch"),
    ("bin_trunc_not_floor", "float f = floorf(u);", "float f = (float)(int)u;", "bins"),
    ("bin_linear_transposed", "return ((long)uz * nb[1] + uy) * nb[0] + ux;", "return ((long)ux * nb[1] + uy) * nb[0] + uz;", "bins"),
    ("bin_margin_m_minus_1", "double m = ceil(c / b);", "double m = floor(c / b);", "bins"),
    ("pad_charge", "slot[3] = 0.0f;", "slot[3] = 1.0f;", "bins"),
    ("bin_unstable_order", "for (long a = 0; a < n_atoms; ++a) { /* ascending index: stable */",
     "for (long a = n_atoms - 1; a >= 0; --a) { /* ascending index: stable */", "bins"),
    ("binned_no_margin", "if (!(g2 < reach * reach)) continue;", "if (!(g2 < c->c * c->c * 0.8)) continue;", "bins"),
]


def _run_group_with(so_path: str, group: str) -> list:
    """Run one pin group against another oracle build; names of failing pins."""
    failures = []
    with oracle.use_library(so_path):
        for pin in PINS[group]:
            try:
                pin()
            except (AssertionError, ValueError):  # a pin noticed the slip
                failures.append(pin.__name__)
    return failures


@pytest.mark.parametrize("name,old,new,group", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, group):
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / f"mut_{name}.c"
    mutated.write_text(src.replace(old, new, 1))
    so = oracle.build(str(mutated), str(tmp_path))
    # a child process: a mutant may also crash (an out-of-range bin index),
    # which counts as caught and must not take the test session down
    code = (
        "import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
        "import test_oracle_pins as t\n"
        "f = t._run_group_with(%r, %r)\n"
        "print('FAILED_PINS', ','.join(f))\n"
        "sys.exit(0 if f else 3)\n"
    ) % (os.path.dirname(os.path.abspath(__file__)), os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
         str(so), group)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert proc.returncode != 3, f"mutant {name} survived every {group} pin:\n{proc.stdout}{proc.stderr}"
