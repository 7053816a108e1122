"""fp64 oracle of the long-range part of a multilevel summation -- TEST
INFRASTRUCTURE (only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it; the product never imports it).

The Input Binning lecture's slide "Large Bin Cut-off Kernel Code" (24) names
its cutoff kernel ``mgpot_shortrng_energy`` and sums q (1/r - g(r)) for
r < c with g(r) = GC0 + r^2 (GC1 + r^2 GC2): the short-range part of a
multilevel summation of 1/r.  The pages stop there.  What is left of 1/r
beyond that short-range part is the smooth kernel

    g_c(r) = (1/c) gamma(r/c),   gamma(s) = 15/8 - 5/4 s^2 + 3/8 s^4  (s < 1),
                                 gamma(s) = 1/s                       (s >= 1),

so that V(x) = V_short(x) + V_long(x) exactly, with
V_long(x) = sum_a q_a g_c(|x - r_a|) (``long_range_exact``: the plain
definition, evaluated as the direct sum minus the cutoff sum).

``long_range`` approximates V_long the multilevel way (R. D. Skeel,
I. Tezcan, D. J. Hardy, "Multiple grid methods for classical molecular
dynamics", J. Comput. Chem. 23 (2002); D. J. Hardy, J. E. Stone,
K. Schulten, "Multilevel summation of electrostatic potentials using
graphics processing units", Parallel Computing 35 (2009)), in these steps:

  lattices   level l has spacing h_l = 2^l h0 and nodes o + i h_l, all
             levels sharing the origin o (the low corner of the domain);
  splitting  g_c = sum_{l<L} (g_{2^l c} - g_{2^(l+1) c}) + g_{2^L c}; the
             level-l piece vanishes beyond 2^(l+1) c;
  basis      phi(t) = (1 - |t|)(1 + |t| - 3/2 t^2)  for |t| <= 1,
             phi(t) = -1/2 (|t| - 1)(2 - |t|)^2     for 1 <= |t| <= 2,
             0 beyond (the C1 cubic interpolant), Phi = phi x phi x phi;
  anterpolation  q0_i = sum_a q_a Phi((r_a - o)/h0 - i);
  restriction    q(l+1)_J = sum_i Phi(i/2 - J) q(l)_i;
  lattice cutoff e(l)_i = sum_j K_l(i - j) q(l)_j with
             K_l(d) = g_{2^l c}(|d| h_l) - g_{2^(l+1) c}(|d| h_l) for l < L
             and the dense top level K_L(d) = g_{2^L c}(|d| h_L);
  prolongation  e(l)_i += sum_J Phi(i/2 - J) e(l+1)_J, from the top down;
  interpolation V_long(x) = sum_i Phi((x - o)/h0 - i) e(0)_i.

Every step is written out in numpy float64 in that order, with no blocking
or reordering beyond what numpy's array operations do.

Lattice geometry (the reading adopted where the papers leave a choice):
the domain is the box given by the caller, widened to contain the map's
grid points; level 0 has nc = floor((hi - o)/h0) + 2 cells per axis (one
spare) and the nodes their points need, i = -1 .. nc + 1; level l+1 spans
floor(lo_l/2) - 1 .. ceil(hi_l/2) + 1; the top level L is the first whose
every axis has at most ``top_nodes`` nodes.

Parity: pinned by the tests in tests/test_oracle_msm.py -- phi's partition
of unity and polynomial reproduction, restriction as the exact transpose of
prolongation, prolongation of quadratics, the splitting's telescoping sum,
V_short + V_long_exact = V_direct, and V_long against V_long_exact within
the error the method's interpolation order implies, shrinking as h0 does.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

TOP_NODES = 12
MAX_LEVELS = 16


def gamma(s):
    """The C2 Taylor softening of 1/s: polynomial inside s < 1, 1/s outside."""
    s = np.asarray(s, dtype=np.float64)
    inner = 15.0 / 8.0 - 1.25 * s * s + 0.375 * s ** 4
    with np.errstate(divide="ignore"):
        outer = 1.0 / s
    return np.where(s < 1.0, inner, outer)


def g_smooth(r, c):
    """g_c(r) = gamma(r/c)/c: the long-range kernel left after the switched
    short-range term q (1/r - g(r)), r < c, is taken out of 1/r."""
    return gamma(np.asarray(r, dtype=np.float64) / c) / c


def phi(t):
    """The C1 cubic interpolating basis function (support |t| < 2)."""
    t = np.abs(np.asarray(t, dtype=np.float64))
    near = (1.0 - t) * (1.0 + t - 1.5 * t * t)
    far = -0.5 * (t - 1.0) * (2.0 - t) ** 2
    return np.where(t <= 1.0, near, np.where(t <= 2.0, far, 0.0))


@dataclass
class Level:
    lo: Tuple[int, int, int]  # lowest node index per axis
    n: Tuple[int, int, int]  # nodes per axis
    h: float  # spacing


@dataclass
class Geometry:
    origin: np.ndarray  # lattice origin o (fp64 of the domain's low corner)
    h0: float
    cutoff: float
    levels: List[Level]  # levels[0] .. levels[L]; the last is the top
    cells: Tuple[int, int, int]  # level-0 cells per axis


def geometry(shape, origin, h, domain_lo, domain_hi, cutoff, h0, top_nodes: int = TOP_NODES) -> Geometry:
    """Lattice levels for a map grid (shape, origin, h) inside a domain box."""
    origin = np.asarray(origin, dtype=np.float32).astype(np.float64)
    h = float(np.float32(h))
    h0 = float(np.float32(h0))
    cutoff = float(np.float32(cutoff))
    dlo = np.asarray(domain_lo, dtype=np.float32).astype(np.float64)
    dhi = np.asarray(domain_hi, dtype=np.float32).astype(np.float64)
    gmax = origin + (np.asarray(shape, dtype=np.float64) - 1.0) * h
    lo = np.minimum(dlo, origin)
    hi = np.maximum(dhi, gmax)
    o = lo
    cells = [int(math.floor((hi[k] - o[k]) / h0)) + 2 for k in range(3)]
    top = [cells[k] + 1 for k in range(3)]
    lvl_lo = [-1, -1, -1]
    lvl_hi = top
    levels = []
    hl = h0
    for _ in range(MAX_LEVELS):
        n = tuple(lvl_hi[k] - lvl_lo[k] + 1 for k in range(3))
        levels.append(Level(tuple(lvl_lo), n, hl))
        if max(n) <= top_nodes:
            break
        lvl_lo = [(lvl_lo[k] // 2) - 1 for k in range(3)]
        lvl_hi = [-((-lvl_hi[k]) // 2) + 1 for k in range(3)]
        hl *= 2.0
    return Geometry(o, h0, cutoff, levels, tuple(cells))


def _weights_1d(t0: np.ndarray):
    """For coordinates t0 (in lattice units, relative to node 0), the four
    node indices floor(t0) - 1 .. floor(t0) + 2 and their phi weights."""
    k = np.floor(t0).astype(np.int64)
    idx = k[:, None] + np.arange(-1, 3)[None, :]
    w = phi(t0[:, None] - idx)
    return idx, w


def anterpolate(atoms, geo: Geometry) -> np.ndarray:
    """q0_i = sum_a q_a Phi((r_a - o)/h0 - i) on level 0 (array [nz][ny][nx])."""
    lv = geo.levels[0]
    a = np.asarray(atoms, dtype=np.float32).astype(np.float64)
    q0 = np.zeros(lv.n[::-1], dtype=np.float64)
    ix, wx = _weights_1d((a[:, 0] - geo.origin[0]) / geo.h0)
    iy, wy = _weights_1d((a[:, 1] - geo.origin[1]) / geo.h0)
    iz, wz = _weights_1d((a[:, 2] - geo.origin[2]) / geo.h0)
    for cz in range(4):
        for cy in range(4):
            for cx in range(4):
                w = a[:, 3] * wx[:, cx] * wy[:, cy] * wz[:, cz]
                np.add.at(q0, (iz[:, cz] - lv.lo[2], iy[:, cy] - lv.lo[1], ix[:, cx] - lv.lo[0]), w)
    return q0


def _transfer_matrix(fine: Level, coarse: Level, axis: int) -> np.ndarray:
    """P[i, J] = phi(i/2 - J) for fine nodes i and coarse nodes J of one axis."""
    i = fine.lo[axis] + np.arange(fine.n[axis])
    J = coarse.lo[axis] + np.arange(coarse.n[axis])
    return phi(i[:, None] / 2.0 - J[None, :])


def restrict(q: np.ndarray, fine: Level, coarse: Level) -> np.ndarray:
    """q(l+1)_J = sum_i Phi(i/2 - J) q(l)_i."""
    Px, Py, Pz = (_transfer_matrix(fine, coarse, k) for k in range(3))
    t = np.einsum("zyx,xX->zyX", q, Px)  # one axis at a time
    t = np.einsum("zyX,yY->zYX", t, Py)
    return np.einsum("zYX,zZ->ZYX", t, Pz)


def prolong(e: np.ndarray, fine: Level, coarse: Level) -> np.ndarray:
    """(P e)_i = sum_J Phi(i/2 - J) e_J: the coarse values interpolated to
    the fine nodes."""
    Px, Py, Pz = (_transfer_matrix(fine, coarse, k) for k in range(3))
    t = np.einsum("ZYX,xX->ZYx", e, Px)  # one axis at a time
    t = np.einsum("ZYx,yY->Zyx", t, Py)
    return np.einsum("Zyx,zZ->zyx", t, Pz)


def stencil(geo: Geometry) -> Tuple[np.ndarray, int]:
    """W(d) = g_c(|d| h0) - g_{2c}(|d| h0) on the cube |d_k| <= R (zero
    where |d| h0 >= 2c); level l < L uses 2^-l W."""
    c, h0 = geo.cutoff, geo.h0
    R = int(math.ceil(2.0 * c / h0))
    d = np.arange(-R, R + 1, dtype=np.float64)
    r = h0 * np.sqrt(d[:, None, None] ** 2 + d[None, :, None] ** 2 + d[None, None, :] ** 2)
    W = g_smooth(r, c) - g_smooth(r, 2.0 * c)
    W[r >= 2.0 * c] = 0.0
    return W, R


def lattice_cutoff(q: np.ndarray, W: np.ndarray, R: int, scale: float) -> np.ndarray:
    """e_i = scale * sum_d W(d) q_{i+d} (q is zero outside its lattice)."""
    nz, ny, nx = q.shape
    qp = np.zeros((nz + 2 * R, ny + 2 * R, nx + 2 * R))
    qp[R:R + nz, R:R + ny, R:R + nx] = q
    e = np.zeros_like(q)
    for dz in range(-R, R + 1):
        for dy in range(-R, R + 1):
            for dx in range(-R, R + 1):
                w = W[dz + R, dy + R, dx + R]
                if w != 0.0:
                    e += w * qp[R + dz:R + dz + nz, R + dy:R + dy + ny, R + dx:R + dx + nx]
    return scale * e


def top_level(q: np.ndarray, lv: Level, c_top: float) -> np.ndarray:
    """Dense top level: e_i = sum_j g_{c_top}(|x_i - x_j|) q_j."""
    nz, ny, nx = q.shape
    zz, yy, xx = np.meshgrid(np.arange(nz), np.arange(ny), np.arange(nx), indexing="ij")
    pos = lv.h * np.stack([xx.ravel(), yy.ravel(), zz.ravel()], axis=1)
    diff = pos[:, None, :] - pos[None, :, :]
    K = g_smooth(np.sqrt((diff * diff).sum(axis=2)), c_top)
    return (K @ q.ravel()).reshape(q.shape)


def lattice_potentials(atoms, geo: Geometry) -> List[np.ndarray]:
    """Every level's lattice potential e(l) after prolongation (e(0) first)."""
    L = len(geo.levels) - 1
    qs = [anterpolate(atoms, geo)]
    for l in range(L):
        qs.append(restrict(qs[l], geo.levels[l], geo.levels[l + 1]))
    es: List[Optional[np.ndarray]] = [None] * (L + 1)
    es[L] = top_level(qs[L], geo.levels[L], geo.cutoff * 2.0 ** L)
    W, R = stencil(geo)
    for l in range(L - 1, -1, -1):
        es[l] = lattice_cutoff(qs[l], W, R, 2.0 ** -l) + prolong(es[l + 1], geo.levels[l], geo.levels[l + 1])
    return es


def interpolate(e0: np.ndarray, geo: Geometry, xyz: np.ndarray) -> np.ndarray:
    """V_long(x) = sum_i Phi((x - o)/h0 - i) e(0)_i at points xyz (m, 3)."""
    lv = geo.levels[0]
    ix, wx = _weights_1d((xyz[:, 0] - geo.origin[0]) / geo.h0)
    iy, wy = _weights_1d((xyz[:, 1] - geo.origin[1]) / geo.h0)
    iz, wz = _weights_1d((xyz[:, 2] - geo.origin[2]) / geo.h0)
    v = np.zeros(len(xyz))
    for cz in range(4):
        for cy in range(4):
            for cx in range(4):
                v += wx[:, cx] * wy[:, cy] * wz[:, cz] * e0[iz[:, cz] - lv.lo[2], iy[:, cy] - lv.lo[1],
                                                          ix[:, cx] - lv.lo[0]]
    return v


def grid_positions(shape, origin, h, points: Optional[np.ndarray] = None) -> np.ndarray:
    """fp64 coordinates origin + (i, j, k) h of the map points (all, x
    fastest, or the listed (i, j, k) rows)."""
    origin = np.asarray(origin, dtype=np.float32).astype(np.float64)
    h = float(np.float32(h))
    if points is None:
        nx, ny, nz = shape
        k, j, i = np.meshgrid(np.arange(nz), np.arange(ny), np.arange(nx), indexing="ij")
        points = np.stack([i.ravel(), j.ravel(), k.ravel()], axis=1)
    return origin[None, :] + np.asarray(points, dtype=np.float64) * h


def long_range(atoms, shape, origin, h, domain_lo, domain_hi, cutoff, h0, points=None,
               top_nodes: int = TOP_NODES) -> np.ndarray:
    """Multilevel approximation of V_long at the map points (all, x fastest,
    or the listed (i, j, k) rows)."""
    geo = geometry(shape, origin, h, domain_lo, domain_hi, cutoff, h0, top_nodes)
    es = lattice_potentials(atoms, geo)
    return interpolate(es[0], geo, grid_positions(shape, origin, h, points))


def long_range_exact(atoms, shape, origin, h, cutoff, points=None) -> np.ndarray:
    """V_long(x) = sum_a q_a g_c(|x - r_a|) written out directly."""
    a = np.asarray(atoms, dtype=np.float32).astype(np.float64)
    xyz = grid_positions(shape, origin, h, points)
    c = float(np.float32(cutoff))
    out = np.empty(len(xyz))
    step = max(1, 2_000_000 // max(1, len(a)))
    for s in range(0, len(xyz), step):
        d = xyz[s:s + step, None, :] - a[None, :, :3]
        r = np.sqrt((d * d).sum(axis=2))
        out[s:s + step] = (g_smooth(r, c) * a[None, :, 3]).sum(axis=1)
    return out


def abs_charge_bound(atoms, shape, origin, h, cutoff, points=None) -> np.ndarray:
    """sum_a |q_a| g_c(|x - r_a|): the scale the method's error is measured on."""
    a = np.asarray(atoms, dtype=np.float32).astype(np.float64).copy()
    a[:, 3] = np.abs(a[:, 3])
    return long_range_exact(a, shape, origin, h, cutoff, points)
