"""fp64 CPU oracle for electrostatic potential maps -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or runs it, and it never imports the
product: the two share only the seeded input generators of ``workloads``.

The arithmetic lives in ``oracle.c`` (plain C, double precision, compiled
here with gcc on first use); this module only marshals numpy arrays.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  direct         pinned: closed forms (single charge, symmetric shells,
                 dipole), scipy cdist special case, linearity, translation.
  cutoff_brute   pinned: switched-term closed forms (g(c)=1/c, slope and
                 curvature match at c), large-c limit to the direct sum plus
                 the constant shift, cdist special case, mutant detection.
  cutoff_binned  pinned: bit-identical V and pair set against cutoff_brute.
  cutoff_hard    pinned: large-c limit equals direct exactly term by term,
                 single-charge closed forms inside and outside c, cdist
                 special case, mutant detection.
  bin_atoms      pinned: numpy float32 re-derivation of every bin index,
                 counts, permutation, pad layout.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None

PAD_COORD = np.float32(1.0e18)

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]


def _src_hash(path: str, extra: str = "") -> str:
    with open(path, "rb") as f:
        return hashlib.sha1(f.read() + extra.encode()).hexdigest()[:12]


def build(src: str = _SRC, out_dir: str = _BUILD, force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``_build/liboracle-<hash>.so``."""
    os.makedirs(out_dir, exist_ok=True)
    tag = _src_hash(src, " ".join(CFLAGS))
    base = os.path.splitext(os.path.basename(src))[0]
    so = os.path.join(out_dir, f"lib{base}-{tag}.so")
    if force or not os.path.exists(so):
        tmp = so + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, so)
    return so


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; returns a ctypes CDLL."""
    global _LIB
    with _LOCK:
        if path is None and _LIB is not None:
            return _LIB
        lib = ctypes.CDLL(path or build())
        _declare(lib)
        if path is None:
            _LIB = lib
        return lib


class use_library:
    """Context manager: route every wrapper through another build of the
    oracle (the mutation tests compile deliberately broken copies)."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _LIB
        lib = load(self.path)
        with _LOCK:
            self.saved = _LIB
            _LIB = lib
        return lib

    def __exit__(self, *exc):
        global _LIB
        with _LOCK:
            _LIB = self.saved
        return False


_P = ctypes.c_void_p
_L = ctypes.c_long
_I = ctypes.c_int
_F = ctypes.c_float
_D = ctypes.c_double
_LL = ctypes.c_longlong


def _declare(lib):
    lib.or_direct.argtypes = [_P, _L, _P, _L, _I, _I, _I, _P, _F, _P, _P, _I]
    lib.or_direct.restype = _I
    lib.or_cutoff_brute.argtypes = [_P, _L, _P, _L, _I, _I, _I, _P, _F, _F, _P, _P, _I]
    lib.or_cutoff_brute.restype = _I
    lib.or_cutoff_hard.argtypes = [_P, _L, _P, _L, _I, _I, _I, _P, _F, _F, _P, _P, _I]
    lib.or_cutoff_hard.restype = _I
    lib.or_cutoff_binned.argtypes = [_P, _L, _P, _L, _I, _I, _I, _P, _F, _F, _F, _P, _P, _I]
    lib.or_cutoff_binned.restype = _I
    lib.or_switch_g.argtypes = [_D, _D]
    lib.or_switch_g.restype = _D
    lib.or_switched_term.argtypes = [_D, _D]
    lib.or_switched_term.restype = _D
    lib.or_bin_geometry.argtypes = [_I, _I, _I, _P, _F, _F, _F, _P, _P, _P]
    lib.or_bin_geometry.restype = _I
    lib.or_atom_bin.argtypes = [_P, _P, _P, _F]
    lib.or_atom_bin.restype = _L
    lib.or_bin_atoms.argtypes = [_P, _L, _P, _P, _F, _I, _P, _P, _P, _P, _P, _P, _P]
    lib.or_bin_atoms.restype = _L
    lib.or_pairs_brute.argtypes = [_P, _L, _P, _L, _I, _I, _I, _P, _F, _F, _P, _LL]
    lib.or_pairs_brute.restype = _LL
    lib.or_pairs_binned.argtypes = [_P, _L, _P, _L, _I, _I, _I, _P, _F, _F, _F, _P, _LL]
    lib.or_pairs_binned.restype = _LL


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _atoms(atoms) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(atoms, dtype=np.float32))
    if a.ndim != 2 or a.shape[1] != 4:
        raise ValueError("atoms must be (n, 4) float32")
    return a


def _pts(points) -> Optional[np.ndarray]:
    if points is None:
        return None
    p = np.ascontiguousarray(np.asarray(points, dtype=np.int32))
    if p.ndim != 2 or p.shape[1] != 3:
        raise ValueError("points must be (m, 3) int32 (i, j, k)")
    return p


def _origin(origin) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(origin, dtype=np.float32).reshape(3))


def _npts(shape, pts) -> int:
    return int(pts.shape[0]) if pts is not None else int(shape[0]) * int(shape[1]) * int(shape[2])


def direct(atoms, shape, origin, h, points=None, threads: Optional[int] = None, with_bound: bool = True):
    """fp64 direct sum V(g) = sum_a q_a / r at the listed (or all) grid points.

    Returns (V, B): float64 arrays, B = sum |q_a|/r.  With ``points=None`` the
    arrays are the whole grid in x-fastest order (flat; reshape to (Nz, Ny, Nx)).
    """
    lib = load()
    a, p, o = _atoms(atoms), _pts(points), _origin(origin)
    m = _npts(shape, p)
    V = np.empty(m, dtype=np.float64)
    B = np.empty(m, dtype=np.float64) if with_bound else None
    rc = lib.or_direct(_ptr(a), a.shape[0], _ptr(p), m, int(shape[0]), int(shape[1]), int(shape[2]),
                       _ptr(o), float(np.float32(h)), _ptr(V), _ptr(B), threads or default_threads())
    if rc != 0:
        raise ValueError(f"or_direct failed ({rc})")
    return V, B


def cutoff_brute(atoms, shape, origin, h, cutoff, points=None, threads: Optional[int] = None, with_bound=True):
    """fp64 switched cutoff sum by brute force over all atoms: (V, B)."""
    lib = load()
    a, p, o = _atoms(atoms), _pts(points), _origin(origin)
    m = _npts(shape, p)
    V = np.empty(m, dtype=np.float64)
    B = np.empty(m, dtype=np.float64) if with_bound else None
    rc = lib.or_cutoff_brute(_ptr(a), a.shape[0], _ptr(p), m, int(shape[0]), int(shape[1]), int(shape[2]),
                             _ptr(o), float(np.float32(h)), float(np.float32(cutoff)), _ptr(V), _ptr(B),
                             threads or default_threads())
    if rc != 0:
        raise ValueError(f"or_cutoff_brute failed ({rc})")
    return V, B


def cutoff_hard(atoms, shape, origin, h, cutoff, points=None, threads: Optional[int] = None, with_bound=True):
    """fp64 hard-cutoff sum (no switching): sum of q/r over r^2 < c^2: (V, B)."""
    lib = load()
    a, p, o = _atoms(atoms), _pts(points), _origin(origin)
    m = _npts(shape, p)
    V = np.empty(m, dtype=np.float64)
    B = np.empty(m, dtype=np.float64) if with_bound else None
    rc = lib.or_cutoff_hard(_ptr(a), a.shape[0], _ptr(p), m, int(shape[0]), int(shape[1]), int(shape[2]),
                            _ptr(o), float(np.float32(h)), float(np.float32(cutoff)), _ptr(V), _ptr(B),
                            threads or default_threads())
    if rc != 0:
        raise ValueError(f"or_cutoff_hard failed ({rc})")
    return V, B


def cutoff_binned(atoms, shape, origin, h, cutoff, bin_size, points=None, threads: Optional[int] = None,
                  with_bound=True):
    """fp64 switched cutoff sum through bins and per-point neighbourhoods: (V, B)."""
    lib = load()
    a, p, o = _atoms(atoms), _pts(points), _origin(origin)
    m = _npts(shape, p)
    V = np.empty(m, dtype=np.float64)
    B = np.empty(m, dtype=np.float64) if with_bound else None
    rc = lib.or_cutoff_binned(_ptr(a), a.shape[0], _ptr(p), m, int(shape[0]), int(shape[1]), int(shape[2]),
                              _ptr(o), float(np.float32(h)), float(np.float32(cutoff)),
                              float(np.float32(bin_size)), _ptr(V), _ptr(B), threads or default_threads())
    if rc != 0:
        raise ValueError(f"or_cutoff_binned failed ({rc})")
    return V, B


def switch_g(r2: float, c: float) -> float:
    return load().or_switch_g(float(r2), float(c))


def switched_term(r2: float, c: float) -> float:
    """1/r - g(r) at r^2 = r2 (no cutoff test)."""
    return load().or_switched_term(float(r2), float(c))


def bin_geometry(shape, origin, h, cutoff, bin_size):
    """(nb[3] int, bo[3] float32, m) of the bin grid for this map."""
    lib = load()
    nb = np.zeros(3, dtype=np.int32)
    bo = np.zeros(3, dtype=np.float32)
    m = ctypes.c_int(0)
    o = _origin(origin)
    rc = lib.or_bin_geometry(int(shape[0]), int(shape[1]), int(shape[2]), _ptr(o), float(np.float32(h)),
                             float(np.float32(cutoff)), float(np.float32(bin_size)), _ptr(nb), _ptr(bo),
                             ctypes.addressof(m))
    if rc != 0:
        raise ValueError(f"or_bin_geometry failed ({rc})")
    return nb, bo, int(m.value)


def bin_atoms(atoms, shape, origin, h, cutoff, bin_size, capacity: int):
    """Stable counting sort into bins (see oracle.c).  Returns a dict with
    nb, bo, bin_of_atom, count, start, csr_index, csr_atoms, padded, n_dropped."""
    lib = load()
    a = _atoms(atoms)
    nb, bo, m = bin_geometry(shape, origin, h, cutoff, bin_size)
    nbins = int(nb[0]) * int(nb[1]) * int(nb[2])
    n = a.shape[0]
    bin_of_atom = np.empty(n, dtype=np.int32)
    count = np.empty(nbins, dtype=np.int32)
    start = np.empty(nbins + 1, dtype=np.int32)
    csr_index = np.empty(max(n, 1), dtype=np.int32)
    csr_atoms = np.empty((max(n, 1), 4), dtype=np.float32)
    padded = np.empty((nbins, max(capacity, 1), 4), dtype=np.float32)
    dropped = ctypes.c_long(0)
    nbinned = lib.or_bin_atoms(_ptr(a), n, _ptr(nb), _ptr(bo), float(np.float32(bin_size)), int(capacity),
                               _ptr(bin_of_atom), _ptr(count), _ptr(start), _ptr(csr_index), _ptr(csr_atoms),
                               _ptr(padded) if capacity > 0 else None, ctypes.addressof(dropped))
    if nbinned < 0:
        raise ValueError(f"or_bin_atoms failed ({nbinned})")
    return {
        "nb": nb,
        "bo": bo,
        "m": m,
        "bin_of_atom": bin_of_atom,
        "count": count,
        "start": start,
        "csr_index": csr_index[:nbinned],
        "csr_atoms": csr_atoms[:nbinned],
        "padded": padded[:, :capacity] if capacity > 0 else padded[:, :0],
        "n_dropped": int(dropped.value),
        "n_binned": int(nbinned),
    }


def _pairs(fn, *args):
    cap = 1 << 16
    while True:
        out = np.empty(2 * cap, dtype=np.int64)
        k = fn(*args, _ptr(out), cap)
        if k < 0:
            raise ValueError(f"pair enumeration failed ({k})")
        if k <= cap:
            return out[: 2 * k].reshape(k, 2)
        cap = int(k)


def pairs_brute(atoms, shape, origin, h, cutoff, points=None) -> np.ndarray:
    """(k, 2) int64 array of contributing (point ordinal, atom index), r^2 < c^2, brute force."""
    lib = load()
    a, p, o = _atoms(atoms), _pts(points), _origin(origin)
    m = _npts(shape, p)
    return _pairs(lib.or_pairs_brute, _ptr(a), a.shape[0], _ptr(p), m, int(shape[0]), int(shape[1]),
                  int(shape[2]), _ptr(o), float(np.float32(h)), float(np.float32(cutoff)))


def pairs_binned(atoms, shape, origin, h, cutoff, bin_size, points=None) -> np.ndarray:
    """Same pair set as ``pairs_brute`` but found through the bins."""
    lib = load()
    a, p, o = _atoms(atoms), _pts(points), _origin(origin)
    m = _npts(shape, p)
    return _pairs(lib.or_pairs_binned, _ptr(a), a.shape[0], _ptr(p), m, int(shape[0]), int(shape[1]),
                  int(shape[2]), _ptr(o), float(np.float32(h)), float(np.float32(cutoff)),
                  float(np.float32(bin_size)))


def tolerance_ok(v_test, v_ref, bound, rel: float = 2e-4):
    """Elementwise |v_test - v_ref| <= rel * bound (bound = sum |q|/r)."""
    v_test = np.asarray(v_test, dtype=np.float64)
    return np.abs(v_test - np.asarray(v_ref)) <= rel * np.asarray(bound)
