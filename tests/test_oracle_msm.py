"""Pins of the multilevel long-range oracle (oracle/msm.py) to facts that do
not come from the oracle itself: the cubic basis's interpolation and
polynomial reproduction, restriction as the exact transpose of
prolongation, moment conservation of anterpolation, the switching identity
against the C oracle's switched term, V_short + V_long = V_direct against
the C oracle's direct and cutoff sums, and the multilevel error against the
exact long-range sum, falling like h0^3.  Each pin is also run on planted
mistakes (a wrong basis, a transposed transfer, a flipped stencil sign, a
dropped level) and must fail there."""
import contextlib

import numpy as np
import pytest

import oracle
import workloads
from oracle import msm



# ---------------------------------------------------------------------------
# pins written as functions returning (ok, detail), so that mutants can be
# checked against the same code


def pin_basis():
    rng = np.random.default_rng(11)
    t = rng.uniform(-5.0, 5.0, 2000)
    i = np.arange(-10, 11)
    w = msm.phi(t[:, None] - i[None, :])
    ok = np.allclose(w.sum(1), 1.0, atol=1e-13)  # partition of unity
    ok &= np.allclose((w * i).sum(1), t, atol=1e-12)  # linear reproduction
    ok &= np.allclose((w * i * i).sum(1), t * t, atol=1e-11)  # quadratic reproduction
    # interpolating: phi(0) = 1, phi(+-1) = phi(+-2) = 0; C1 at |t| = 1
    ok &= float(msm.phi(0.0)) == 1.0 and float(msm.phi(1.0)) == 0.0 and float(msm.phi(2.0)) == 0.0
    e = 1e-7
    d_in = (msm.phi(1.0 - e) - msm.phi(1.0 - 2 * e)) / e
    d_out = (msm.phi(1.0 + 2 * e) - msm.phi(1.0 + e)) / e
    ok &= abs(d_in - d_out) < 1e-5
    return bool(ok), "basis"


def pin_switching():
    """g_c(r) + the C oracle's switched term q(1/r - g(r)) = 1/r for r < c; g_c
    = 1/r beyond c; gamma is C2 at s = 1."""
    c = 12.0
    r = np.linspace(0.3, 11.99, 200)
    s = np.array([oracle.switched_term(float(x * x), c) for x in r])
    ok = np.allclose(msm.g_smooth(r, c) + s, 1.0 / r, rtol=1e-13, atol=0)
    rr = np.linspace(12.0, 40.0, 50)
    ok &= np.allclose(msm.g_smooth(rr, c), 1.0 / rr, rtol=1e-15)
    # value, slope and curvature of gamma at 1 from both sides
    e = 1e-4
    f = lambda x: float(msm.gamma(x))
    ok &= abs(f(1.0) - 1.0) < 1e-15
    slope_in = (f(1.0) - f(1.0 - e)) / e
    slope_out = (f(1.0 + e) - f(1.0)) / e
    ok &= abs(slope_in + 1.0) < 1e-3 and abs(slope_out + 1.0) < 1e-3
    curv_in = (f(1.0) - 2 * f(1.0 - e) + f(1.0 - 2 * e)) / e ** 2
    curv_out = (f(1.0 + 2 * e) - 2 * f(1.0 + e) + f(1.0)) / e ** 2
    ok &= abs(curv_in - 2.0) < 1e-2 and abs(curv_out - 2.0) < 1e-2
    return bool(ok), "switching"


def _two_levels():
    geo = msm.geometry((30, 26, 22), (0.0, 0.0, 0.0), 0.5, (-3.0, -2.0, -1.0), (17.0, 15.0, 12.0), 3.0, 0.5)
    assert len(geo.levels) >= 2
    return geo, geo.levels[0], geo.levels[1]


def pin_transfer_adjoint():
    """<P e, q>_fine = <e, R q>_coarse for random e, q."""
    geo, F, C = _two_levels()
    rng = np.random.default_rng(12)
    q = rng.normal(size=F.n[::-1])
    e = rng.normal(size=C.n[::-1])
    lhs = float((msm.prolong(e, F, C) * q).sum())
    rhs = float((e * msm.restrict(q, F, C)).sum())
    return abs(lhs - rhs) <= 1e-10 * (abs(lhs) + 1.0), f"adjoint {lhs} {rhs}"


def pin_prolong_quadratic():
    """Prolongation of a quadratic on the coarse nodes reproduces it on the
    fine nodes whose coarse stencil lies inside the coarse lattice."""
    geo, F, C = _two_levels()

    def quad(lv):
        z, y, x = np.meshgrid(*[lv.lo[k] + np.arange(lv.n[k]) for k in (2, 1, 0)], indexing="ij")
        X, Y, Z = x * lv.h, y * lv.h, z * lv.h
        return 0.3 + 0.1 * X - 0.2 * Y + 0.05 * Z + 0.01 * X * Y - 0.02 * Z * Z + 0.015 * X * X

    got = msm.prolong(quad(C), F, C)
    want = quad(F)
    sl = tuple(slice(4, -4) for _ in range(3))
    return bool(np.allclose(got[sl], want[sl], atol=1e-11)), "prolong quadratic"


def _small_system(seed=21, n=300):
    rng = np.random.default_rng(seed)
    pos = rng.uniform(-4.0, 14.0, size=(n, 3))
    q = rng.uniform(-1.0, 1.0, size=n)
    return np.concatenate([pos, q[:, None]], axis=1).astype(np.float32)


def pin_anterp_moments():
    """sum_i q0_i p(x_i) = sum_a q_a p(r_a) for p of degree <= 2."""
    atoms = _small_system()
    a = atoms.astype(np.float64)
    geo = msm.geometry((20, 20, 20), (0.0, 0.0, 0.0), 0.5, a[:, :3].min(0), a[:, :3].max(0), 3.0, 1.0)
    q0 = msm.anterpolate(atoms, geo)
    lv = geo.levels[0]
    z, y, x = np.meshgrid(*[lv.lo[k] + np.arange(lv.n[k]) for k in (2, 1, 0)], indexing="ij")
    X = geo.origin[0] + x * geo.h0
    Y = geo.origin[1] + y * geo.h0
    Z = geo.origin[2] + z * geo.h0
    ok = True
    for fl, fa in ((lambda: np.ones_like(X), lambda: np.ones(len(a))),
                   (lambda: X, lambda: a[:, 0]), (lambda: Y * Z, lambda: a[:, 1] * a[:, 2]),
                   (lambda: X * X, lambda: a[:, 0] ** 2)):
        lhs = float((q0 * fl()).sum())
        rhs = float((a[:, 3] * fa()).sum())
        ok &= abs(lhs - rhs) <= 1e-9 * (1.0 + np.abs(a[:, 3]).sum() * 400)
    return bool(ok), "anterpolation moments"


def pin_interp_quadratic():
    geo, F, C = _two_levels()
    z, y, x = np.meshgrid(*[F.lo[k] + np.arange(F.n[k]) for k in (2, 1, 0)], indexing="ij")
    X, Y, Z = (geo.origin[k] + v * geo.h0 for k, v in enumerate((x, y, z)))
    p = lambda X, Y, Z: 1.0 + 0.2 * X - 0.1 * Y * Y + 0.03 * X * Z
    e0 = p(X, Y, Z)
    rng = np.random.default_rng(13)
    xyz = rng.uniform(0.0, 10.0, size=(500, 3)) + geo.origin[None, :]
    got = msm.interpolate(e0, geo, xyz)
    return bool(np.allclose(got, p(xyz[:, 0], xyz[:, 1], xyz[:, 2]), atol=1e-11)), "interpolation"


def pin_stencil_single_charge():
    """A unit charge on one level-0 node: the level-0 lattice cutoff gives
    W(i - j) = g_c(|d| h0) - g_2c(|d| h0), zero from 2c on."""
    geo = msm.geometry((16, 16, 16), (0.0, 0.0, 0.0), 0.5, (0.0, 0.0, 0.0), (7.5, 7.5, 7.5), 2.0, 0.5)
    lv = geo.levels[0]
    W, R = msm.stencil(geo)
    q = np.zeros(lv.n[::-1])
    j = (lv.n[2] // 2, lv.n[1] // 2, lv.n[0] // 2)
    q[j] = 1.0
    e = msm.lattice_cutoff(q, W, R, 1.0)
    z, y, x = np.meshgrid(*[np.arange(lv.n[k]) for k in (2, 1, 0)], indexing="ij")
    r = geo.h0 * np.sqrt((x - j[2]) ** 2 + (y - j[1]) ** 2 + (z - j[0]) ** 2)
    want = np.where(r < 2 * geo.cutoff, 1.0 / geo.cutoff * (msm.gamma(r / geo.cutoff) - 0.5 * msm.gamma(r / (2 * geo.cutoff))), 0.0)
    return bool(np.allclose(e, want, atol=1e-14)), "stencil"


def _accuracy_case():
    w = workloads.random_case(7, 400, (20, 18, 16), h=0.5, origin=(0.0, 0.0, 0.0), margin=6.0, cutoff=4.0,
                              bin_size=2.0)
    pts = workloads.sample_points(w.shape, 200, seed=5)
    lo, hi = w.atoms[:, :3].min(0), w.atoms[:, :3].max(0)
    exact = msm.long_range_exact(w.atoms, w.shape, w.origin, w.h, w.cutoff, points=pts)
    bound = msm.abs_charge_bound(w.atoms, w.shape, w.origin, w.h, w.cutoff, points=pts)
    return w, pts, lo, hi, exact, bound


_ACC = {}


def pin_accuracy():
    """Multilevel error against the exact long-range sum, relative to
    sum |q| g_c: below 4e-3 at c/h0 = 2, 6e-4 at c/h0 = 4, 8e-5 at c/h0 = 8,
    and falling by at least 5x per halving of h0 (third order: 8x)."""
    if "case" not in _ACC:
        _ACC["case"] = _accuracy_case()
    w, pts, lo, hi, exact, bound = _ACC["case"]
    errs = []
    for h0 in (2.0, 1.0, 0.5):
        v = msm.long_range(w.atoms, w.shape, w.origin, w.h, lo, hi, w.cutoff, h0, points=pts)
        errs.append(float((np.abs(v - exact) / bound).max()))
    ok = errs[0] < 4e-3 and errs[1] < 6e-4 and errs[2] < 8e-5
    ok &= errs[0] / errs[1] > 5.0 and errs[1] / errs[2] > 5.0
    return bool(ok), f"errors {errs}"


PINS = [pin_basis, pin_switching, pin_transfer_adjoint, pin_prolong_quadratic, pin_anterp_moments,
        pin_interp_quadratic, pin_stencil_single_charge, pin_accuracy]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_msm_oracle_pin(pin):
    ok, detail = pin()
    assert ok, detail


def test_decomposition_is_exact():
    """V_direct = V_short (switched cutoff sum) + V_long exactly, with the C
    oracle providing the direct and cutoff sums."""
    w = workloads.random_case(8, 300, (14, 12, 10), h=0.5, origin=(1.0, -1.0, 0.5), margin=5.0, cutoff=3.0,
                              bin_size=1.5)
    vd, _ = oracle.direct(w.atoms, w.shape, w.origin, w.h)
    vs, _ = oracle.cutoff_brute(w.atoms, w.shape, w.origin, w.h, w.cutoff)
    vl = msm.long_range_exact(w.atoms, w.shape, w.origin, w.h, w.cutoff)
    assert np.allclose(vs + vl, vd, rtol=0, atol=1e-12 * np.abs(vd).max())


def test_geometry_covers_atoms_and_grid():
    w = workloads.random_case(9, 200, (25, 9, 13), h=0.4, origin=(-2.0, 3.0, 1.0), margin=7.0, cutoff=3.0,
                              bin_size=1.5)
    lo, hi = w.atoms[:, :3].min(0), w.atoms[:, :3].max(0)
    geo = msm.geometry(w.shape, w.origin, w.h, lo, hi, w.cutoff, 0.7)
    lv = geo.levels[0]
    xyz = np.concatenate([w.atoms[:, :3].astype(np.float64), msm.grid_positions(w.shape, w.origin, w.h)])
    t = (xyz - geo.origin[None, :]) / geo.h0
    k = np.floor(t).astype(int)
    for d in range(3):
        assert (k[:, d] - 1 >= lv.lo[d]).all() and (k[:, d] + 2 <= lv.lo[d] + lv.n[d] - 1).all()
        assert (k[:, d] >= 0).all() and (k[:, d] < geo.cells[d]).all()
    assert max(geo.levels[-1].n) <= msm.TOP_NODES
    for a, b in zip(geo.levels, geo.levels[1:]):
        assert all(b.n[d] < a.n[d] for d in range(3)) and b.h == 2 * a.h


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail


@contextlib.contextmanager
def _patched(name, value):
    old = getattr(msm, name)
    setattr(msm, name, value)
    try:
        _ACC.clear()
        yield
    finally:
        setattr(msm, name, old)
        _ACC.clear()


def _hat(t):  # linear interpolation instead of the cubic
    t = np.abs(np.asarray(t, dtype=np.float64))
    return np.where(t < 1.0, 1.0 - t, 0.0)


def _bad_transfer(fine, coarse, axis):  # phi(i/2 - J) with the sign of the offset flipped on odd nodes
    i = fine.lo[axis] + np.arange(fine.n[axis])
    J = coarse.lo[axis] + np.arange(coarse.n[axis])
    return msm.phi((i[:, None] + (i[:, None] % 2)) / 2.0 - J[None, :])


_orig_stencil = msm.stencil
_orig_lattice_potentials = msm.lattice_potentials
_orig_gamma = msm.gamma


def _neg_stencil(geo):
    W, R = _orig_stencil(geo)
    return -W, R


def _drop_top(atoms, geo):  # forget the top level's contribution
    es = _orig_lattice_potentials(atoms, geo)
    L = len(geo.levels) - 1
    if L == 0:
        return [np.zeros_like(es[0])]
    zero = [np.zeros_like(e) for e in es]
    # recompute without the top: every level's own lattice cutoff only
    W, R = _orig_stencil(geo)
    qs = [msm.anterpolate(atoms, geo)]
    for l in range(L):
        qs.append(msm.restrict(qs[l], geo.levels[l], geo.levels[l + 1]))
    zero[L - 1] = msm.lattice_cutoff(qs[L - 1], W, R, 2.0 ** -(L - 1))
    for l in range(L - 2, -1, -1):
        zero[l] = msm.lattice_cutoff(qs[l], W, R, 2.0 ** -l) + msm.prolong(zero[l + 1], geo.levels[l], geo.levels[l + 1])
    return zero


def _gamma_wrong_quartic(s):
    s = np.asarray(s, dtype=np.float64)
    inner = 15.0 / 8.0 - 1.25 * s * s + 0.5 * s ** 4
    with np.errstate(divide="ignore"):
        outer = 1.0 / s
    return np.where(s < 1.0, inner, outer)


MUTANTS = {
    "linear_basis": ("phi", _hat),
    "transfer_offset": ("_transfer_matrix", _bad_transfer),
    "stencil_sign": ("stencil", _neg_stencil),
    "no_top_level": ("lattice_potentials", _drop_top),
    "gamma_quartic": ("gamma", _gamma_wrong_quartic),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_msm_mutant_is_caught(mutant):
    name, value = MUTANTS[mutant]
    with _patched(name, value):
        failed = [p.__name__ for p in PINS if not p()[0]]
    assert failed, f"mutant {mutant} passed every pin"
