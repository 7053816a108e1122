"""CPU tests of the C ABI: the library loads, exports every symbol the
header declares, rejects bad arguments on the host before any launch, and
its host logic (bin geometry, workspace layout, brick offset list) agrees
with the independent oracle and with the pages' figures."""
import ctypes
import json
import math
import os
import re

import numpy as np
import pytest

import direct_coulomb_summation_gb300 as cp
from direct_coulomb_summation_gb300 import _lib
import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpmap.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "page_figures.json")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CP_API\s+[\w\s\*]+?\b(cp_\w+)\s*\(", text)))


def test_header_symbols_exported():
    names = declared_symbols()
    assert len(names) >= 13
    lib = cp.library()
    for name in names:
        assert hasattr(lib, name), f"{name} declared in cpmap.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"
    # and nothing exported by the binding is undeclared
    assert set(_lib.SIGNATURES) == set(names)


def test_library_is_in_tree_and_built_for_sm103a():
    path = _lib.library_path()
    assert os.path.commonpath([path, ROOT]) == ROOT
    assert os.path.exists(path)
    from direct_coulomb_summation_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.NVCC_FLAGS)


def test_status_strings():
    assert cp.status_string(0) == "ok"
    for code in range(-7, 0):
        assert cp.status_string(code) != "unknown status"
    assert cp.version() >= 100


GRID = [4, 4, 4, _lib.cp_vec3(0.0, 0.0, 0.0), 0.5]
FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: the calls return first
FAKE_MIS = ctypes.c_void_p(0x10004)  # 4-byte aligned only


@pytest.mark.parametrize("args,code", [
    ((FAKE, -1, *GRID, FAKE, None), -1),                                  # negative atom count
    ((None, 5, *GRID, FAKE, None), -1),                                   # null atoms
    ((FAKE, 5, *GRID, None, None), -1),                                   # null V
    ((FAKE, 5, 0, 4, 4, GRID[3], 0.5, FAKE, None), -1),                   # empty grid
    ((FAKE, 5, 4, 4, 4, GRID[3], 0.0, FAKE, None), -1),                   # h = 0
    ((FAKE, 5, 4, 4, 4, GRID[3], float("nan"), FAKE, None), -1),          # h NaN
    ((FAKE, 5, 4, 4, 4, _lib.cp_vec3(float("inf"), 0, 0), 0.5, FAKE, None), -1),
    ((FAKE_MIS, 5, *GRID, FAKE, None), -2),                               # atoms not 16-B aligned
    ((FAKE, 5, 1 << 25, 1, 1, GRID[3], 0.5, FAKE, None), -3),             # axis beyond 2^24
    ((FAKE, 5, 2048, 2048, 1024, GRID[3], 0.5, FAKE, None), -3),          # 2^32 points
])
def test_direct_rejects_on_host(args, code):
    assert cp.library().cp_direct(*args) == code


def test_direct_config_rejects_bad_variant():
    lib = cp.library()
    assert lib.cp_direct_config(FAKE, 5, *GRID, FAKE, len(cp.DIRECT_VARIANTS), 0, None) == -1
    assert lib.cp_direct_config(FAKE, 5, *GRID, FAKE, 0, 17, None) == -1
    assert lib.cp_direct_config(FAKE, 5, *GRID, FAKE, 0, -2, None) == -1


def test_cutoff_rejects_on_host():
    lib = cp.library()
    n, c, b = 10, 12.0, 4.0
    need = lib.cp_cutoff_workspace_bytes(n, *GRID, c, b, 16)
    assert need > 0
    ws = ctypes.c_void_p(0x100000)
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, 16, ws, need, FAKE, None) != -4  # would launch: no GPU here
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, 16, ws, need - 1, FAKE, None) == -4
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, 12, ws, need, FAKE, None) == -5   # capacity
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, -8, ws, need, FAKE, None) == -5
    assert lib.cp_cutoff(FAKE, n, *GRID, -1.0, b, 16, ws, need, FAKE, None) == -1
    assert lib.cp_cutoff(FAKE, n, *GRID, c, 0.0, 16, ws, need, FAKE, None) == -1
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, 16, ctypes.c_void_p(0x100010), need, FAKE, None) == -2
    assert lib.cp_cutoff(FAKE_MIS, n, *GRID, c, b, 16, ws, need, FAKE, None) == -2
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, 16, None, need, FAKE, None) == -1
    assert lib.cp_cutoff(FAKE, n, *GRID, c, b, 16, ws, need, None, None) == -1
    assert lib.cp_cutoff(FAKE, n, *GRID, c, 1e-6, 16, ws, need, FAKE, None) == -3  # huge bin grid
    assert lib.cp_cutoff_workspace_bytes(n, *GRID, c, b, 12) == 0


@pytest.mark.parametrize("shape,origin,h,c,b", [
    ((200, 200, 200), (0.0, 0.0, 0.0), 0.5, 12.0, 4.0),
    ((400, 400, 400), (0.0, 0.0, 0.0), 0.5, 12.0, 4.0),
    ((37, 21, 9), (-3.25, 1.5, 100.0), 0.37, 5.5, 1.75),
    ((8, 8, 1), (0.0, 0.0, 5.0), 0.5, 2.0, 4.0),
])
def test_bin_geometry_matches_oracle(shape, origin, h, c, b):
    L = cp.cutoff_layout(1000, shape, origin, h, c, b, 16)
    nb, bo, m = oracle.bin_geometry(shape, origin, h, c, b)
    assert list(L.nb) == list(nb)
    assert np.array_equal(np.array(list(L.bo), dtype=np.float32), bo)
    assert L.margin_bins == m
    assert L.nbins == int(np.prod(nb))
    offs = [L.off_count, L.off_start, L.off_csr_index, L.off_csr_atoms, L.off_padded, L.off_stats, L.off_scratch]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert L.off_padded + 16 * L.nbins * 16 <= L.off_stats < L.total_bytes


def test_offset_list_page_efficiency():
    """Brick neighbourhood for 8x8x8 points at h = 0.5, 4 A bins, c = 12 A: the
    share of the examined volume inside the cutoff sphere matches the page's figure."""
    fig = json.load(open(GOLDEN))["small_bin_examined_within_cutoff"]
    geo = fig["geometry"]
    runs = cp.offset_list((200, 200, 200), (0, 0, 0), geo["h"], geo["cutoff"], geo["bin_size"])
    n_bins = int((runs[:, 3] - runs[:, 2] + 1).sum())
    # for uniform atoms the brick's 512 cutoff spheres all lie inside the listed
    # bins, so the expected share is the sphere volume over the listed volume
    share = (4.0 / 3.0) * math.pi * geo["cutoff"] ** 3 / (n_bins * geo["bin_size"] ** 3)
    assert abs(share - fig["value"]) <= fig["tolerance"], (n_bins, share)
    # the 27-bin scheme of PMPP ch.18 notes section 18.5 (bins of edge c) examines
    # 27 c^3 per point: far less efficient
    assert share > 2 * (4.0 / 3.0) * math.pi / 27


def test_offset_list_runs_wellformed():
    runs = cp.offset_list((200, 200, 200), (0, 0, 0), 0.5, 12.0, 4.0)
    assert len(runs) > 0
    assert np.all(runs[:, 3] >= runs[:, 2])
    # one run per (dy, dz) row
    assert len({(int(a), int(b)) for a, b in runs[:, :2]}) == len(runs)
    # the home bin and its face neighbours are always listed
    def listed(dx, dy, dz):
        sel = (runs[:, 0] == dy) & (runs[:, 1] == dz)
        return bool(np.any((runs[sel, 2] <= dx) & (dx <= runs[sel, 3])))
    for d in [(0, 0, 0), (1, 0, 0), (-1, 0, 0), (0, 1, 0), (0, -1, 0), (0, 0, 1), (0, 0, -1)]:
        assert listed(*d)
    # aligned case (brick points span 3.5 A of a 4 A bin): bin dx = +4 starts
    # 12.5 A past the brick and is left out; bin dx = -4 ends exactly 12 A
    # before it and is kept, because an atom rounded into it by the fp32 bin
    # rule can lie a hair inside the cutoff; dx = -5 is out
    assert listed(-4, 0, 0) and not listed(-5, 0, 0) and not listed(4, 0, 0)


@pytest.mark.parametrize("seed,shape,origin,h,c,b", [
    (1, (24, 20, 17), (0.0, 0.0, 0.0), 0.5, 3.0, 1.0),
    (2, (19, 23, 16), (-2.1, 0.7, 3.3), 0.4, 2.5, 1.3),
    (3, (16, 16, 16), (0.0, 0.0, 0.0), 0.5, 4.0, 4.0),
    (4, (21, 9, 30), (10.0, -5.0, 0.25), 0.3, 1.9, 0.55),
])
def test_offset_list_covers_every_contributing_pair(seed, shape, origin, h, c, b):
    """Every (point, atom) pair with r < c (found by the oracle's brute force)
    has its atom, binned by the oracle's fp32 rule, in a bin of the point's
    brick neighbourhood (home bin + listed offsets)."""
    w = workloads.random_case(seed, 400, shape, h=h, origin=origin, margin=c + b)
    runs = cp.offset_list(shape, origin, h, c, b)
    res = oracle.bin_atoms(w.atoms, shape, origin, h, c, b, capacity=0)
    nb = res["nb"]
    bins = res["bin_of_atom"]
    pairs = oracle.pairs_brute(w.atoms, shape, origin, h, c)
    assert len(pairs) > 1000
    pts = workloads.grid_points(shape)
    homes = {}
    for p, a in pairs:
        i, j, k = pts[p]
        brick = (i // 8, j // 8, k // 8)
        if brick not in homes:
            homes[brick] = cp.brick_home(shape, origin, h, c, b, brick)
        hx, hy, hz = homes[brick]
        bi = int(bins[a])
        assert bi >= 0, "a contributing atom was dropped by the bin rule"
        ux, uy, uz = bi % nb[0], (bi // nb[0]) % nb[1], bi // (nb[0] * nb[1])
        dx, dy, dz = ux - hx, uy - hy, uz - hz
        sel = (runs[:, 0] == dy) & (runs[:, 1] == dz)
        assert np.any((runs[sel, 2] <= dx) & (dx <= runs[sel, 3])), (p, a, (dx, dy, dz))


def test_brick_home_contains_brick_origin():
    shape, origin, h, c, b = (64, 40, 33), (-1.0, 2.0, 0.5), 0.45, 3.0, 1.6
    nb, bo, m = oracle.bin_geometry(shape, origin, h, c, b)
    for brick in [(0, 0, 0), (3, 2, 1), (7, 4, 4)]:
        home = cp.brick_home(shape, origin, h, c, b, brick)
        for d in range(3):
            lo = float(np.float32(origin[d])) + 8 * brick[d] * float(np.float32(h))
            blo = float(bo[d]) + home[d] * float(np.float32(b))
            assert blo - 1e-4 <= lo < blo + float(np.float32(b)) + 1e-4


def test_cutoff_rejects_huge_cutoff_to_bin_ratio():
    lib = cp.library()
    # more than 127 margin bins, or an offset list longer than the kernels take
    assert lib.cp_cutoff_workspace_bytes(10, *GRID, 200.0, 1.0, 0) == 0
    nr, nb = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.cp_offset_list(*GRID, 40.0, 1.0, None, 0, ctypes.byref(nr), ctypes.byref(nb)) == -3
    ws = ctypes.c_void_p(0x100000)
    assert lib.cp_cutoff(FAKE, 10, *GRID, 200.0, 1.0, 0, ws, 1 << 30, FAKE, None) == -3


# ---------------------------------------------------------------------------
# multilevel long-range part: host geometry against the oracle's rule

from oracle import msm as msm_oracle  # noqa: E402

MSM_CASES = [
    # shape, origin, h, domain_lo, domain_hi, c, h0
    ((200, 200, 200), (0.0, 0.0, 0.0), 0.5, (0.0, 0.0, 0.0), (100.0, 100.0, 100.0), 12.0, 2.0),
    ((400, 400, 400), (0.0, 0.0, 0.0), 0.5, (0.0, 0.0, 0.0), (200.0, 200.0, 200.0), 12.0, 2.5),
    ((37, 21, 19), (-1.0, 0.5, 2.0), 0.5, (-6.2, -4.0, -3.1), (22.0, 15.5, 16.0), 4.0, 0.7),
    ((8, 8, 8), (0.0, 0.0, 0.0), 0.5, (0.0, 0.0, 0.0), (4.0, 4.0, 4.0), 2.0, 1.0),
    ((30, 5, 9), (3.0, 3.0, 3.0), 0.25, (10.0, 10.0, 10.0), (11.0, 11.0, 11.0), 3.0, 0.6),  # grid outside the box
]


@pytest.mark.parametrize("shape,origin,h,lo,hi,c,h0", MSM_CASES)
def test_msm_geometry_matches_oracle(shape, origin, h, lo, hi, c, h0):
    L = cp.msm_layout(1000, shape, origin, h, c, h0, (lo, hi))
    geo = msm_oracle.geometry(shape, origin, h, lo, hi, c, h0)
    assert L.levels == len(geo.levels)
    for l, lv in enumerate(geo.levels):
        assert tuple(L.lo[l]) == lv.lo and tuple(L.n[l]) == lv.n
    assert tuple(L.cells) == geo.cells
    assert (L.lattice_origin.x, L.lattice_origin.y, L.lattice_origin.z) == tuple(np.float32(geo.origin))
    W, R = msm_oracle.stencil(geo)
    assert L.radius == R and L.taps == int((W != 0).sum())
    assert max(L.n[L.levels - 1]) <= 12
    assert L.total_bytes == cp.msm_workspace_bytes(1000, shape, origin, h, c, h0, (lo, hi))
    offs = sorted([L.off_cells, L.off_stencil] + [L.off_q[l] for l in range(L.levels)] +
                  [L.off_e[l] for l in range(L.levels)])
    assert all(o % 256 == 0 for o in offs) and len(set(offs)) == len(offs) and offs[-1] < L.total_bytes
    assert L.off_partial % 256 == 0 and offs[-1] < L.off_partial <= L.total_bytes  # empty with one level


def test_msm_rejects_on_host():
    lib = cp.library()
    lo, hi = _lib.cp_vec3(0.0, 0.0, 0.0), _lib.cp_vec3(100.0, 100.0, 100.0)
    args = (10, *GRID, lo, hi)
    need = lib.cp_msm_workspace_bytes(*args, 12.0, 2.0)
    assert need > 0
    ws = ctypes.c_void_p(0x100000)
    call = lambda c, h0, ws_=ws, n=need, V=FAKE, acc=0, lo_=lo, hi_=hi, atoms=FAKE: lib.cp_msm_longrange(
        atoms, 10, *GRID, lo_, hi_, c, h0, ws_, n, V, acc, None)
    assert call(12.0, 2.0, n=need - 1) == -4
    assert call(12.0, 0.0) == -1 and call(-1.0, 2.0) == -1 and call(float("nan"), 2.0) == -1
    assert call(12.0, 0.9) == -3  # stencil radius ceil(24/0.9) = 27 > 24
    assert lib.cp_msm_workspace_bytes(*args, 12.0, 0.9) == 0
    assert call(12.0, 2.0, hi_=_lib.cp_vec3(-1.0, 100.0, 100.0)) == -1  # domain hi < lo
    assert call(12.0, 2.0, acc=2) == -1
    assert call(12.0, 2.0, V=None) == -1
    assert call(12.0, 2.0, ws_=ctypes.c_void_p(0x100010)) == -2
    assert call(12.0, 2.0, atoms=FAKE_MIS) == -2
    assert lib.cp_atom_bounds(FAKE, 0, FAKE, None) == -1
    assert lib.cp_atom_bounds(FAKE_MIS, 5, FAKE, None) == -2


def _axis_exact_brute(o, h, n):
    o64, h64 = float(np.float32(o)), float(np.float32(h))
    v = o64 + np.arange(n, dtype=np.float64) * h64
    return bool(np.all(v.astype(np.float32).astype(np.float64) == v))


@pytest.mark.parametrize("seed", range(6))
def test_grid_points_exact_is_sound(seed):
    """cp_grid_points_exact (which picks the kernels' difference form) never
    claims exact fp32 grid points that are not, checked point by point; it
    recognises the dyadic benchmark grids; and it rejects an invalid grid."""
    lib = cp.library()
    rng = np.random.default_rng(seed)
    hs = [0.5, 0.25, 0.37, 0.1, 1.0, 0.3, 0.125, 2.0 ** -10]
    for _ in range(60):
        n = [int(v) for v in rng.integers(1, 400, size=3)]
        h = float(np.float32(hs[rng.integers(len(hs))]))
        kind = rng.integers(3)
        scale = [1.0, 100.0, 1e5][rng.integers(3)]
        if kind == 0:
            o = [float(np.float32(np.round(v * 4) / 4)) for v in rng.uniform(-scale, scale, 3)]
        elif kind == 1:
            o = [float(np.float32(v)) for v in rng.uniform(-scale, scale, 3)]
        else:
            o = [0.0, 0.0, float(np.float32(10 * h))]
        got = lib.cp_grid_points_exact(*n, _lib.cp_vec3(*o), h)
        assert got in (0, 1)
        brute = all(_axis_exact_brute(o[d], h, n[d]) for d in range(3))
        if got == 1:
            assert brute, (n, o, h)
    for shape, origin in [((128, 128, 64), (0, 0, 0)), ((200, 200, 200), (0, 0, 0)), ((100, 100, 1), (0, 0, 5.0)),
                          ((400, 400, 400), (0, 0, 0))]:
        assert lib.cp_grid_points_exact(*shape, _lib.cp_vec3(*origin), 0.5) == 1
    assert lib.cp_grid_points_exact(20, 14, 11, _lib.cp_vec3(5000.1234567, -4999.2345679, 2500.31415), 0.37) == 0
    assert lib.cp_grid_points_exact(0, 4, 4, _lib.cp_vec3(0, 0, 0), 0.5) == -1
