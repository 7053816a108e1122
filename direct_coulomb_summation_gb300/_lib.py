"""ctypes view of libcpmap.so: symbol declarations and nothing else.

Every declaration mirrors one in ``include/cpmap.h``.  The library is the
product's only compute path; if it cannot be built or loaded this module
raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LOCK = threading.Lock()
_LIB = None


class cp_vec3(ctypes.Structure):
    _fields_ = [("x", ctypes.c_float), ("y", ctypes.c_float), ("z", ctypes.c_float)]


class cp_cutoff_layout(ctypes.Structure):
    _fields_ = [
        ("nb", ctypes.c_int * 3),
        ("bo", ctypes.c_float * 3),
        ("margin_bins", ctypes.c_int),
        ("capacity", ctypes.c_int),
        ("nbins", ctypes.c_longlong),
        ("off_count", ctypes.c_size_t),
        ("off_start", ctypes.c_size_t),
        ("off_csr_index", ctypes.c_size_t),
        ("off_csr_atoms", ctypes.c_size_t),
        ("off_padded", ctypes.c_size_t),
        ("off_stats", ctypes.c_size_t),
        ("off_scratch", ctypes.c_size_t),
        ("total_bytes", ctypes.c_size_t),
    ]


class cp_cutoff_stats_t(ctypes.Structure):
    _fields_ = [
        ("n_binned", ctypes.c_int),
        ("n_dropped", ctypes.c_int),
        ("n_overflow", ctypes.c_int),
        ("max_bin_count", ctypes.c_int),
    ]


MSM_MAX_LEVELS = 16


class cp_msm_layout(ctypes.Structure):
    _fields_ = [
        ("levels", ctypes.c_int),
        ("lo", (ctypes.c_int * 3) * MSM_MAX_LEVELS),
        ("n", (ctypes.c_int * 3) * MSM_MAX_LEVELS),
        ("split", ctypes.c_int * MSM_MAX_LEVELS),
        ("radius", ctypes.c_int),
        ("taps", ctypes.c_int),
        ("cells", ctypes.c_int * 3),
        ("lattice_origin", cp_vec3),
        ("q_dims", (ctypes.c_int * 3) * MSM_MAX_LEVELS),
        ("q_plane", ctypes.c_int * MSM_MAX_LEVELS),
        ("off_q", ctypes.c_size_t * MSM_MAX_LEVELS),
        ("off_e", ctypes.c_size_t * MSM_MAX_LEVELS),
        ("off_cells", ctypes.c_size_t),
        ("off_stencil", ctypes.c_size_t),
        ("off_partial", ctypes.c_size_t),
        ("total_bytes", ctypes.c_size_t),
    ]


_I, _F, _P, _SZ = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_GRID = [_I, _I, _I, cp_vec3, _F]  # nx, ny, nz, origin, h

SIGNATURES = {
    "cp_direct": (_I, [_P, _I, *_GRID, _P, _P]),
    "cp_direct_config": (_I, [_P, _I, *_GRID, _P, _I, _I, _P]),
    "cp_direct_plan": (_I, [_I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "cp_grid_points_exact": (_I, [_I, _I, _I, cp_vec3, _F]),
    "cp_cutoff_layout_of": (_I, [_I, *_GRID, _F, _F, _I, ctypes.POINTER(cp_cutoff_layout)]),
    "cp_cutoff_workspace_bytes": (_SZ, [_I, *_GRID, _F, _F, _I]),
    "cp_cutoff": (_I, [_P, _I, *_GRID, _F, _F, _I, _P, _SZ, _P, _P]),
    "cp_bin_atoms": (_I, [_P, _I, *_GRID, _F, _F, _I, _P, _SZ, _P]),
    "cp_cutoff_map": (_I, [_P, _I, *_GRID, _F, _F, _I, _P, _SZ, _P, _P]),
    "cp_launch_count": (ctypes.c_ulonglong, []),
    "cp_cutoff_pair_counts": (_I, [_P, _I, *_GRID, _F, _F, _I, _P, _SZ, _P, _P]),
    "cp_cutoff_no_alloc": (_I, [_P, _I, *_GRID, _F, _F, _I, _P, _P]),
    "cp_cutoff_stats": (_I, [_P, _SZ, _I, *_GRID, _F, _F, _I, ctypes.POINTER(cp_cutoff_stats_t), _P]),
    "cp_offset_list": (_I, [*_GRID, _F, _F, _P, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "cp_brick_home": (_I, [*_GRID, _F, _F, _I, _I, _I, _I * 3]),
    "cp_device_status": (_I, [ctypes.POINTER(ctypes.c_uint), _P]),
    "cp_status_string": (ctypes.c_char_p, [_I]),
    "cp_version": (_I, []),
    "cp_eval_rsqrt": (_I, [_I, _P, _P, _I, _P]),
    "cp_direct_variant": (_I, [_I, _P, _I, *_GRID, _P, _P]),
    "cp_cutoff27_workspace_bytes": (_SZ, [_I, *_GRID, _F]),
    "cp_cutoff27": (_I, [_P, _I, *_GRID, _F, _P, _SZ, _P, _P]),
    "cp_probe_pipe_rate": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), _P]),
    "cp_msm_layout_of": (_I, [_I, *_GRID, cp_vec3, cp_vec3, _F, _F, ctypes.POINTER(cp_msm_layout)]),
    "cp_msm_workspace_bytes": (_SZ, [_I, *_GRID, cp_vec3, cp_vec3, _F, _F]),
    "cp_msm_longrange": (_I, [_P, _I, *_GRID, cp_vec3, cp_vec3, _F, _F, _P, _SZ, _P, _I, _P]),
    "cp_atom_bounds": (_I, [_P, _I, _P, _P]),
    "cp_probe_wait_timeout": (_I, [ctypes.c_ulonglong, _P, _P]),
    "cp_slab": (_I, [_I, _I, _I, _I, _F, _F, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_F)]),
}


def checked() -> bool:
    """True when CPMAP_CHECKED=1 selects the bounds-checked build."""
    return os.environ.get("CPMAP_CHECKED", "") == "1"


def library_path() -> str:
    return _build.LIB_CHECKED if checked() else _build.LIB


def load(auto_build: bool = True):
    """The loaded libcpmap.so (built first if missing or stale)."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        if not _build.up_to_date(checked()):
            if not auto_build:
                raise RuntimeError(f"{os.path.basename(library_path())} is missing or stale; "
                                   "run direct_coulomb_summation_gb300.build")
            _build.build(checked=checked())
        lib = ctypes.CDLL(library_path())
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
        return lib


def loaded_path():
    return _build.LIB if _LIB is not None else None
