"""Seeded synthetic inputs for electrostatic potential maps.

This module only draws random inputs: atom positions and charges, grid
shapes and sampled grid points.  It holds none of the potential-map
arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA path
(``direct_coulomb_summation_gb300``) can use it without sharing any of the
method's code.

Atoms are returned as a C-contiguous ``float32`` array of shape ``(n, 4)``
holding ``(x, y, z, q)`` per atom, the 16-byte record the pages use for an
atom (PMPP ch.18 notes, section 18.2, ``struct Atom``).  Grid point
``(i, j, k)`` sits at ``origin + (i*h, j*h, k*h)``.

Positions are kept off the grid lattice: every coordinate's fractional
offset from the lattice lies in ``[0.1, 0.9] * h``, so no atom sits on a
grid point and ``1/r`` stays finite (closest approach ``sqrt(3)*0.05*h``).

The five named workloads follow the benchmark described on the pwwt.cn
PMPP chapter-18 article (section 一: a 100x100x50 grid at 0.5 A, 10 000
random atoms, only the z=10 plane) and larger direct and cutoff maps of the
same kind (a 200^3 protein-sized map as in PMPP ch.18 notes section 18.1).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "make",
    "random_case",
    "off_lattice_uniform",
    "sample_points",
    "grid_points",
]


@dataclass
class Workload:
    """One potential-map problem: atoms plus a grid (and cutoff geometry)."""

    name: str
    atoms: np.ndarray  # (n, 4) float32: x, y, z, q
    shape: tuple  # (Nx, Ny, Nz)
    origin: tuple  # 3 x float32 values (as Python floats exactly representable in fp32)
    h: float  # grid spacing, an fp32 value
    cutoff: Optional[float] = None  # None for the direct sum
    bin_size: Optional[float] = None
    description: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def n_atoms(self) -> int:
        return int(self.atoms.shape[0])

    @property
    def n_points(self) -> int:
        nx, ny, nz = self.shape
        return int(nx) * int(ny) * int(nz)

    @property
    def n_pairs(self) -> int:
        return self.n_atoms * self.n_points


def _f32(v) -> float:
    return float(np.float32(v))


def _charges_uniform(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.uniform(-1.0, 1.0, size=n).astype(np.float32)


def _charges_protein(rng: np.random.Generator, n: int) -> np.ndarray:
    values = np.array([-1.0, -0.5, 0.5, 1.0], dtype=np.float32)
    return rng.choice(values, size=n, p=[0.15, 0.35, 0.35, 0.15]).astype(np.float32)


def _lattice_fraction_ok(coord32: np.ndarray, origin: float, h: float) -> np.ndarray:
    """True where the fp32 coordinate sits in [0.1, 0.9]*h of its lattice cell."""
    t = (coord32.astype(np.float64) - origin) / h
    frac = t - np.floor(t)
    return (frac >= 0.1) & (frac <= 0.9)


def off_lattice_uniform(rng, n, lo, hi, origin, h):
    """n positions uniform over the lattice cells of the box [lo, hi) (per axis),

    each coordinate at a fractional offset in [0.1, 0.9]*h of its cell.
    ``lo``/``hi``/``origin`` are 3-sequences; cells are those of the lattice
    ``origin + k*h`` that lie inside the box.
    """
    out = np.empty((n, 3), dtype=np.float32)
    for d in range(3):
        k0 = int(np.ceil((lo[d] - origin[d]) / h - 1e-9))
        k1 = int(np.floor((hi[d] - origin[d]) / h + 1e-9))  # exclusive
        if k1 <= k0:
            raise ValueError("box thinner than one lattice cell")
        cell = rng.integers(k0, k1, size=n)
        frac = rng.uniform(0.1, 0.9, size=n)
        out[:, d] = (origin[d] + (cell + frac) * h).astype(np.float32)
    # fp32 rounding can only move a value by ~1e-7 relative; re-draw the rare
    # coordinate that fell outside the allowed band.
    for d in range(3):
        bad = ~_lattice_fraction_ok(out[:, d], origin[d], h)
        while bad.any():
            m = int(bad.sum())
            k0 = int(np.ceil((lo[d] - origin[d]) / h - 1e-9))
            k1 = int(np.floor((hi[d] - origin[d]) / h + 1e-9))
            cell = rng.integers(k0, k1, size=m)
            frac = rng.uniform(0.15, 0.85, size=m)
            out[bad, d] = (origin[d] + (cell + frac) * h).astype(np.float32)
            bad = ~_lattice_fraction_ok(out[:, d], origin[d], h)
    return out


def _gaussian_clusters_off_lattice(rng, n, centres, sigma, origin, h):
    """n positions from isotropic Gaussians around randomly chosen centres;

    any atom with a coordinate whose lattice fraction is outside [0.1, 0.9]
    is redrawn (same cluster) until all three coordinates are off-lattice.
    """
    which = rng.integers(0, len(centres), size=n)
    pos = np.empty((n, 3), dtype=np.float32)
    todo = np.arange(n)
    while todo.size:
        c = centres[which[todo]]
        p = (c + rng.normal(0.0, sigma, size=(todo.size, 3))).astype(np.float32)
        ok = np.ones(todo.size, dtype=bool)
        for d in range(3):
            ok &= _lattice_fraction_ok(p[:, d], origin[d], h)
        pos[todo[ok]] = p[ok]
        todo = todo[~ok]
    return pos


def _pack(pos: np.ndarray, q: np.ndarray) -> np.ndarray:
    atoms = np.empty((pos.shape[0], 4), dtype=np.float32)
    atoms[:, :3] = pos
    atoms[:, 3] = q
    return np.ascontiguousarray(atoms)


def _ball_uniform(rng, n, centre, radius):
    v = rng.normal(size=(n, 3))
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    r = radius * rng.uniform(0.0, 1.0, size=n) ** (1.0 / 3.0)
    return np.asarray(centre, dtype=np.float64) + v * r[:, None]


def direct_plane(seed: int = 1001) -> Workload:
    """100x100 plane (z-index 10 of a 100x100x50 grid, h = 0.5 A), 10 000 atoms."""
    rng = np.random.default_rng(seed)
    h = 0.5
    origin = (0.0, 0.0, _f32(10 * h))
    lattice0 = (0.0, 0.0, 0.0)
    pos = off_lattice_uniform(rng, 10_000, (0, 0, 0), (50.0, 50.0, 25.0), lattice0, h)
    return Workload(
        name="direct_plane_100x100_10k",
        atoms=_pack(pos, _charges_uniform(rng, 10_000)),
        shape=(100, 100, 1),
        origin=origin,
        h=h,
        description="direct sum, z-index 10 plane of a 100x100x50 grid at h=0.5 A, "
        "10,000 off-lattice atoms uniform in [0,50)x[0,50)x[0,25) A, q~U[-1,1]",
    )


def direct_3d(seed: int = 1002) -> Workload:
    """128x128x64 grid at h = 0.5 A, 40 000 atoms uniform in the box."""
    rng = np.random.default_rng(seed)
    h = 0.5
    origin = (0.0, 0.0, 0.0)
    pos = off_lattice_uniform(rng, 40_000, (0, 0, 0), (64.0, 64.0, 32.0), origin, h)
    return Workload(
        name="direct_3d_128x128x64_40k",
        atoms=_pack(pos, _charges_uniform(rng, 40_000)),
        shape=(128, 128, 64),
        origin=origin,
        h=h,
        description="direct sum, 128x128x64 grid at h=0.5 A (1,048,576 points), "
        "40,000 off-lattice atoms uniform in the 64x64x32 A box, q~U[-1,1]",
    )


def direct_protein(seed: int = 1003) -> Workload:
    """200^3 grid at h = 0.5 A; 100 000 atoms in 200 Gaussian clusters (sigma 3 A)."""
    rng = np.random.default_rng(seed)
    h = 0.5
    origin = (0.0, 0.0, 0.0)
    centres = _ball_uniform(rng, 200, (50.0, 50.0, 50.0), 30.0)
    pos = _gaussian_clusters_off_lattice(rng, 100_000, centres, 3.0, origin, h)
    return Workload(
        name="direct_protein_200^3_100k",
        atoms=_pack(pos, _charges_protein(rng, 100_000)),
        shape=(200, 200, 200),
        origin=origin,
        h=h,
        description="direct sum, 200^3 grid at h=0.5 A, 100,000 off-lattice atoms from 200 "
        "Gaussian clusters (sigma 3 A) centred in a 30 A ball at (50,50,50), "
        "q in {-1,-0.5,0.5,1} w.p. {.15,.35,.35,.15}",
    )


def cutoff_uniform(seed: int = 1004) -> Workload:
    """200^3 grid at h = 0.5 A, 100 000 atoms uniform in [0,100)^3, c = 12 A, 4 A bins."""
    rng = np.random.default_rng(seed)
    h = 0.5
    origin = (0.0, 0.0, 0.0)
    pos = off_lattice_uniform(rng, 100_000, (0, 0, 0), (100.0, 100.0, 100.0), origin, h)
    return Workload(
        name="cutoff_uniform_200^3_100k_c12",
        atoms=_pack(pos, _charges_uniform(rng, 100_000)),
        shape=(200, 200, 200),
        origin=origin,
        h=h,
        cutoff=12.0,
        bin_size=4.0,
        description="cutoff sum c=12 A, 200^3 grid at h=0.5 A, 100,000 off-lattice atoms "
        "uniform in [0,100)^3 A, q~U[-1,1], 4 A bins, 8x8x8-point bricks",
    )


def cutoff_large(seed: int = 1005) -> Workload:
    """400^3 grid at h = 0.5 A; 560 000 uniform + 240 000 clustered atoms (500 clusters, sigma 2 A)."""
    rng = np.random.default_rng(seed)
    h = 0.5
    origin = (0.0, 0.0, 0.0)
    uni = off_lattice_uniform(rng, 560_000, (0, 0, 0), (200.0, 200.0, 200.0), origin, h)
    centres = rng.uniform(0.0, 200.0, size=(500, 3))
    clu = _gaussian_clusters_off_lattice(rng, 240_000, centres, 2.0, origin, h)
    pos = np.concatenate([uni, clu], axis=0)
    perm = rng.permutation(pos.shape[0])
    pos = pos[perm]
    return Workload(
        name="cutoff_large_400^3_800k_c12",
        atoms=_pack(pos, _charges_uniform(rng, pos.shape[0])),
        shape=(400, 400, 400),
        origin=origin,
        h=h,
        cutoff=12.0,
        bin_size=4.0,
        description="cutoff sum c=12 A, 400^3 grid at h=0.5 A, 800,000 off-lattice atoms: "
        "70% uniform in [0,200)^3 A, 30% in 500 Gaussian clusters (sigma 2 A), q~U[-1,1]",
    )


WORKLOADS = {
    "direct_plane": direct_plane,
    "direct_3d": direct_3d,
    "direct_protein": direct_protein,
    "cutoff_uniform": cutoff_uniform,
    "cutoff_large": cutoff_large,
}


def make(name: str, seed: Optional[int] = None) -> Workload:
    fn = WORKLOADS[name]
    return fn() if seed is None else fn(seed)


def random_case(
    seed: int,
    n_atoms: int,
    shape,
    h: float = 0.5,
    origin=(0.0, 0.0, 0.0),
    margin: float = 0.0,
    cutoff: Optional[float] = None,
    bin_size: Optional[float] = None,
    charges: str = "uniform",
) -> Workload:
    """A small seeded case: off-lattice atoms uniform over the grid box widened by

    ``margin`` A on every side (so some atoms may lie outside the grid).
    """
    rng = np.random.default_rng(seed)
    h = _f32(h)
    origin = tuple(_f32(o) for o in origin)
    nx, ny, nz = shape
    lo = [origin[0] - margin, origin[1] - margin, origin[2] - margin]
    hi = [origin[0] + nx * h + margin, origin[1] + ny * h + margin, origin[2] + nz * h + margin]
    if n_atoms > 0:
        pos = off_lattice_uniform(rng, n_atoms, lo, hi, origin, h)
        q = _charges_protein(rng, n_atoms) if charges == "protein" else _charges_uniform(rng, n_atoms)
    else:
        pos = np.zeros((0, 3), dtype=np.float32)
        q = np.zeros((0,), dtype=np.float32)
    return Workload(
        name=f"random_{n_atoms}_{nx}x{ny}x{nz}_s{seed}",
        atoms=_pack(pos, q),
        shape=(int(nx), int(ny), int(nz)),
        origin=origin,
        h=h,
        cutoff=None if cutoff is None else _f32(cutoff),
        bin_size=None if bin_size is None else _f32(bin_size),
    )


def sample_points(shape, n: int, seed: int = 4096) -> np.ndarray:
    """n distinct seeded grid points as an (n, 3) int32 array of (i, j, k)."""
    nx, ny, nz = shape
    total = int(nx) * int(ny) * int(nz)
    rng = np.random.default_rng(seed)
    n = min(n, total)
    flat = np.sort(rng.choice(total, size=n, replace=False))
    return grid_points(shape, flat)


def grid_points(shape, flat_index=None) -> np.ndarray:
    """(i, j, k) int32 indices of the given flat x-fastest indices (all points if None)."""
    nx, ny, nz = shape
    if flat_index is None:
        flat_index = np.arange(int(nx) * int(ny) * int(nz), dtype=np.int64)
    flat_index = np.asarray(flat_index, dtype=np.int64)
    i = flat_index % nx
    j = (flat_index // nx) % ny
    k = flat_index // (nx * ny)
    return np.ascontiguousarray(np.stack([i, j, k], axis=1).astype(np.int32))
