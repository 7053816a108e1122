"""GB300 (sm_103a) electrostatic potential maps behind a C ABI.

Python-side argument marshalling for ``libcpmap.so`` (declared in
``include/cpmap.h``).  PyTorch provides device memory and streams only;
every step of the computation runs in the library's CUDA kernels.

    import direct_coulomb_summation_gb300 as cp
    V = cp.direct(atoms, (nx, ny, nz), origin, h)                 # direct sum
    V = cp.cutoff(atoms, (nx, ny, nz), origin, h, 12.0, 4.0)      # cutoff sum
    V = cp.msm_map(atoms, (nx, ny, nz), origin, h, 12.0, 4.0, 2.0) # cutoff + multilevel long range

``atoms`` is an (n, 4) float32 array of (x, y, z, q).  A CUDA tensor gives a
CUDA result on the current stream (asynchronous); a CPU tensor or numpy
array is copied to the current GPU through pinned memory and the result is
copied back (synchronous) -- the end-to-end path.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import _lib
from ._lib import cp_msm_layout, cp_vec3

__all__ = [
    "CpError",
    "direct",
    "cutoff",
    "cutoff_workspace_bytes",
    "direct_plan",
    "direct_variant",
    "cutoff27",
    "DIRECT_STRATEGIES",
    "cutoff_layout",
    "bin_atoms",
    "cutoff_stats",
    "cutoff_pair_counts",
    "offset_list",
    "brick_home",
    "device_status",
    "probe_pipe_rate",
    "eval_rsqrt",
    "status_string",
    "version",
    "library",
    "DIRECT_VARIANTS",
    "atom_bounds",
    "msm_layout",
    "msm_workspace_bytes",
    "msm_longrange",
    "msm_map",
]

# index -> (PX, PY, PZ, EMU, LS): a patch of PX x-points times PY rows times
# PZ planes, the first EMU of its (PX/2)*PY*PZ point pairs with rsqrt on the
# FMA pipe, shared by LS lanes that take every LS-th atom each.  The 2-point
# (10, 11) and shared-patch (12-18) shapes serve grids too small to fill the
# GPU with 4-point patches.
DIRECT_VARIANTS = {0: (4, 4, 2, 0, 1), 1: (4, 2, 2, 0, 1), 2: (4, 4, 1, 0, 1), 3: (4, 2, 1, 0, 1),
                   4: (4, 1, 1, 0, 1), 5: (4, 4, 2, 4, 1), 6: (4, 4, 2, 5, 1), 7: (4, 2, 2, 2, 1),
                   8: (4, 4, 1, 2, 1), 9: (4, 2, 1, 1, 1), 10: (2, 1, 1, 0, 1), 11: (2, 2, 1, 0, 1),
                   12: (4, 1, 1, 0, 4), 13: (4, 1, 1, 0, 2), 14: (4, 2, 1, 1, 4), 15: (4, 2, 1, 1, 2),
                   16: (4, 2, 1, 1, 8), 17: (4, 2, 2, 2, 4), 18: (4, 4, 1, 2, 4)}


class CpError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        super().__init__(f"{where}: {status_string(code)} ({code})" if where else status_string(code))


def library():
    """The loaded ctypes library (builds it first if needed)."""
    return _lib.load()


def status_string(code: int) -> str:
    return library().cp_status_string(int(code)).decode()


def version() -> int:
    return int(library().cp_version())


def _check(rc: int, where: str):
    if rc != 0:
        raise CpError(rc, where)


def _vec3(v) -> cp_vec3:
    v = [float(np.float32(x)) for x in v]
    return cp_vec3(v[0], v[1], v[2])


def _grid(shape, origin, h):
    nx, ny, nz = (int(s) for s in shape)
    return [nx, ny, nz, _vec3(origin), float(np.float32(h))]


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _as_device_atoms(atoms):
    """(device tensor, was_on_host) for an (n, 4) float32 atom array."""
    if isinstance(atoms, np.ndarray):
        atoms = torch.from_numpy(np.ascontiguousarray(atoms, dtype=np.float32))
    if not isinstance(atoms, torch.Tensor):
        raise TypeError("atoms must be a torch tensor or numpy array of shape (n, 4)")
    if atoms.dim() != 2 or atoms.shape[1] != 4 or atoms.dtype != torch.float32:
        raise ValueError("atoms must have shape (n, 4) and dtype float32")
    if atoms.is_cuda:
        return atoms.contiguous(), False
    host = atoms.contiguous()
    if not host.is_pinned():
        host = host.pin_memory()
    return host.to("cuda", non_blocking=True), True


def _out_tensor(out, shape, device):
    nx, ny, nz = (int(s) for s in shape)
    if out is None:
        return torch.empty((nz, ny, nx), dtype=torch.float32, device=device)
    if not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.numel() == nx * ny * nz):
        raise ValueError("out must be a contiguous float32 CUDA tensor with nx*ny*nz elements")
    return out


def _finish_host(V: torch.Tensor, host_out=None) -> torch.Tensor:
    if host_out is None:
        host_out = torch.empty(V.shape, dtype=torch.float32, pin_memory=True)
    elif host_out.is_cuda or host_out.numel() != V.numel() or host_out.dtype != torch.float32:
        raise ValueError("host_out must be a float32 CPU tensor with nx*ny*nz elements")
    host_out.view(V.shape).copy_(V, non_blocking=host_out.is_pinned())
    torch.cuda.current_stream().synchronize()
    return host_out.view(V.shape)


def direct(atoms, shape, origin, h, out=None, stream=None, variant: int = -1, split: int = 0, host_out=None):
    """Direct Coulomb sum V(g) = sum_a q_a / r over the grid; returns V as (nz, ny, nx).

    ``variant``/``split`` force the kernel's point patch and cluster split
    (see ``DIRECT_VARIANTS``; -1/0 let the library choose).  With host atoms,
    ``host_out`` (ideally pinned) receives the result."""
    lib = library()
    dev_atoms, on_host = _as_device_atoms(atoms)
    V = _out_tensor(out, shape, dev_atoms.device)
    s = _stream(stream)
    n = int(dev_atoms.shape[0])
    if variant == -1 and split == 0:
        rc = lib.cp_direct(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h), V.data_ptr(), s)
    else:
        rc = lib.cp_direct_config(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h), V.data_ptr(),
                                  int(variant), int(split), s)
    _check(rc, "cp_direct")
    return _finish_host(V, host_out) if on_host else V


def direct_plan(n_atoms, shape) -> tuple:
    """(variant, split) that cp_direct picks for this grid and atom count on the current GPU."""
    v, sp = ctypes.c_int(0), ctypes.c_int(0)
    nx, ny, nz = (int(x) for x in shape)
    _check(library().cp_direct_plan(int(n_atoms), nx, ny, nz, ctypes.byref(v), ctypes.byref(sp)), "cp_direct_plan")
    return int(v.value), int(sp.value)


DIRECT_STRATEGIES = {"scatter": 0, "gather": 1, "coarsen": 2, "coalesce": 3}


def direct_variant(strategy: str, atoms, shape, origin, h, out=None, stream=None):
    """The direct map by one of the pages' strategies (comparison kernels):
    "scatter", "gather", "coarsen" or "coalesce".  Device atoms only."""
    lib = library()
    dev_atoms, on_host = _as_device_atoms(atoms)
    V = _out_tensor(out, shape, dev_atoms.device)
    n = int(dev_atoms.shape[0])
    rc = lib.cp_direct_variant(DIRECT_STRATEGIES[strategy], dev_atoms.data_ptr() if n else None, n,
                               *_grid(shape, origin, h), V.data_ptr(), _stream(stream))
    _check(rc, "cp_direct_variant")
    return _finish_host(V) if on_host else V


def cutoff27(atoms, shape, origin, h, cutoff, workspace=None, out=None, stream=None):
    """Hard-cutoff map (sum of q/r over r < c) by the 27-bin kernel (comparison kernel)."""
    lib = library()
    dev_atoms, on_host = _as_device_atoms(atoms)
    n = int(dev_atoms.shape[0])
    need = int(lib.cp_cutoff27_workspace_bytes(n, *_grid(shape, origin, h), float(np.float32(cutoff))))
    if need == 0:
        raise CpError(-1, "cp_cutoff27_workspace_bytes")
    ws = _workspace(workspace, need, dev_atoms.device)
    V = _out_tensor(out, shape, dev_atoms.device)
    rc = lib.cp_cutoff27(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h), float(np.float32(cutoff)),
                         ws.data_ptr(), ws.numel() * ws.element_size(), V.data_ptr(), _stream(stream))
    _check(rc, "cp_cutoff27")
    return _finish_host(V) if on_host else V


def cutoff_layout(n_atoms, shape, origin, h, cutoff, bin_size, capacity: int = 16):
    L = _lib.cp_cutoff_layout()
    rc = library().cp_cutoff_layout_of(int(n_atoms), *_grid(shape, origin, h), float(np.float32(cutoff)),
                                       float(np.float32(bin_size)), int(capacity), ctypes.byref(L))
    _check(rc, "cp_cutoff_layout_of")
    return L


def cutoff_workspace_bytes(n_atoms, shape, origin, h, cutoff, bin_size, capacity: int = 16) -> int:
    return int(cutoff_layout(n_atoms, shape, origin, h, cutoff, bin_size, capacity).total_bytes)


def _workspace(workspace, nbytes, device):
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace


def cutoff(atoms, shape, origin, h, cutoff, bin_size, capacity: int = 16, workspace=None, out=None, stream=None,
           host_out=None):
    """Cutoff sum of q (1/r - g(r)) over r < cutoff through bins; returns V as (nz, ny, nx).

    ``workspace``: optional uint8 CUDA tensor of at least
    ``cutoff_workspace_bytes(...)`` bytes (allocated per call if None)."""
    lib = library()
    dev_atoms, on_host = _as_device_atoms(atoms)
    n = int(dev_atoms.shape[0])
    need = cutoff_workspace_bytes(n, shape, origin, h, cutoff, bin_size, capacity)
    ws = _workspace(workspace, need, dev_atoms.device)
    V = _out_tensor(out, shape, dev_atoms.device)
    rc = lib.cp_cutoff(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h), float(np.float32(cutoff)),
                       float(np.float32(bin_size)), int(capacity), ws.data_ptr(), ws.numel() * ws.element_size(),
                       V.data_ptr(), _stream(stream))
    _check(rc, "cp_cutoff")
    return _finish_host(V, host_out) if on_host else V


_cutoff_sum = cutoff  # msm_map's `cutoff` argument shadows the function


def bin_atoms(atoms, shape, origin, h, cutoff, bin_size, capacity: int = 16, workspace=None, stream=None):
    """Runs only the binning stage; returns tensors viewing the workspace:
    count, start, csr_index, csr_atoms, padded (nbins, K, 4), plus the layout."""
    lib = library()
    dev_atoms, _ = _as_device_atoms(atoms)
    n = int(dev_atoms.shape[0])
    L = cutoff_layout(n, shape, origin, h, cutoff, bin_size, capacity)
    ws = _workspace(workspace, int(L.total_bytes), dev_atoms.device)
    rc = lib.cp_bin_atoms(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h),
                          float(np.float32(cutoff)), float(np.float32(bin_size)), int(capacity), ws.data_ptr(),
                          ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "cp_bin_atoms")
    nbins = int(L.nbins)

    def view(off, count, dtype, shape_):
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return ws[off: off + nbytes].view(dtype).view(shape_)

    return {
        "layout": L,
        "workspace": ws,
        "count": view(L.off_count, nbins, torch.int32, (nbins,)),
        "start": view(L.off_start, nbins + 1, torch.int32, (nbins + 1,)),
        "csr_index": view(L.off_csr_index, n, torch.int32, (n,)),
        "csr_atoms": view(L.off_csr_atoms, 4 * n, torch.float32, (n, 4)),
        "padded": view(L.off_padded, 4 * nbins * capacity, torch.float32, (nbins, capacity, 4)),
    }


def cutoff_pair_counts(atoms, shape, origin, h, cutoff, bin_size, capacity: int = 16, workspace=None, stream=None):
    """(useful, evaluated, examined) pair counts of the cutoff map's traversal (synchronous)."""
    lib = library()
    dev_atoms, _ = _as_device_atoms(atoms)
    n = int(dev_atoms.shape[0])
    need = cutoff_workspace_bytes(n, shape, origin, h, cutoff, bin_size, capacity)
    ws = _workspace(workspace, need, dev_atoms.device)
    counts = torch.zeros(3, dtype=torch.int64, device=dev_atoms.device)
    rc = lib.cp_cutoff_pair_counts(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h),
                                   float(np.float32(cutoff)), float(np.float32(bin_size)), int(capacity),
                                   ws.data_ptr(), ws.numel() * ws.element_size(), counts.data_ptr(), _stream(stream))
    _check(rc, "cp_cutoff_pair_counts")
    c = counts.cpu().tolist()
    return {"useful": c[0], "evaluated": c[1], "examined": c[2]}


def cutoff_stats(workspace, n_atoms, shape, origin, h, cutoff, bin_size, capacity: int = 16, stream=None) -> dict:
    """Counters of the last binning pass on this workspace (synchronises the stream)."""
    st = _lib.cp_cutoff_stats_t()
    rc = library().cp_cutoff_stats(workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                   int(n_atoms), *_grid(shape, origin, h), float(np.float32(cutoff)),
                                   float(np.float32(bin_size)), int(capacity), ctypes.byref(st), _stream(stream))
    _check(rc, "cp_cutoff_stats")
    return {"n_binned": st.n_binned, "n_dropped": st.n_dropped, "n_overflow": st.n_overflow,
            "max_bin_count": st.max_bin_count}


def offset_list(shape, origin, h, cutoff, bin_size) -> np.ndarray:
    """The brick neighbourhood offset list as an (n_runs, 4) int array (dy, dz, dx_lo, dx_hi)."""
    lib = library()
    nr, nb = ctypes.c_int(0), ctypes.c_int(0)
    args = [*_grid(shape, origin, h), float(np.float32(cutoff)), float(np.float32(bin_size))]
    _check(lib.cp_offset_list(*args, None, 0, ctypes.byref(nr), ctypes.byref(nb)), "cp_offset_list")
    runs = np.zeros((max(nr.value, 1), 4), dtype=np.int32)
    _check(lib.cp_offset_list(*args, runs.ctypes.data, nr.value, ctypes.byref(nr), ctypes.byref(nb)),
           "cp_offset_list")
    return runs[: nr.value]


def brick_home(shape, origin, h, cutoff, bin_size, brick) -> tuple:
    out = (ctypes.c_int * 3)()
    rc = library().cp_brick_home(*_grid(shape, origin, h), float(np.float32(cutoff)), float(np.float32(bin_size)),
                                 int(brick[0]), int(brick[1]), int(brick[2]), out)
    _check(rc, "cp_brick_home")
    return tuple(out)


def device_status(stream=None) -> int:
    """Reads and clears the device status word (0 = every kernel finished cleanly)."""
    bits = ctypes.c_uint(0)
    _check(library().cp_device_status(ctypes.byref(bits), _stream(stream)), "cp_device_status")
    return int(bits.value)


PIPE_KINDS = {"mufu_rsqrt": 0, "ffma": 1}


def eval_rsqrt(x: "torch.Tensor", kind: str = "sfu", stream=None) -> "torch.Tensor":
    """rsqrt of a float32 CUDA tensor by the kernels' SFU ("sfu") or FMA-pipe ("fma") route."""
    if not (x.is_cuda and x.dtype == torch.float32):
        raise ValueError("x must be a float32 CUDA tensor")
    x = x.contiguous()
    y = torch.empty_like(x)
    rc = library().cp_eval_rsqrt({"sfu": 0, "fma": 1}[kind], x.data_ptr(), y.data_ptr(), x.numel(), _stream(stream))
    _check(rc, "cp_eval_rsqrt")
    return y


def probe_pipe_rate(kind: str, warps: int = 32, iters: int = 4096, stream=None):
    """(operations per SM clock, kernel ms) of one SM pipe."""
    r, ms = ctypes.c_double(0), ctypes.c_double(0)
    rc = library().cp_probe_pipe_rate(PIPE_KINDS[kind], int(warps), int(iters), ctypes.byref(r), ctypes.byref(ms),
                                      _stream(stream))
    _check(rc, "cp_probe_pipe_rate")
    return float(r.value), float(ms.value)


# ---------------------------------------------------------------------------
# multilevel summation: long-range part


def atom_bounds(atoms, stream=None):
    """The atoms' bounding box ((min x, y, z), (max x, y, z)), computed by the
    library's reduction kernel and read back (synchronises the stream)."""
    lib = library()
    dev_atoms, _ = _as_device_atoms(atoms)
    n = int(dev_atoms.shape[0])
    out = torch.empty(6, dtype=torch.float32, device=dev_atoms.device)
    _check(lib.cp_atom_bounds(dev_atoms.data_ptr(), n, out.data_ptr(), _stream(stream)), "cp_atom_bounds")
    b = out.cpu().numpy()
    return tuple(float(v) for v in b[:3]), tuple(float(v) for v in b[3:])


def _domain(domain, dev_atoms, stream):
    if domain is not None:
        return domain
    if dev_atoms.shape[0] == 0:
        return (0.0, 0.0, 0.0), (0.0, 0.0, 0.0)
    return atom_bounds(dev_atoms, stream)


def msm_layout(n_atoms, shape, origin, h, cutoff, lattice_h, domain) -> cp_msm_layout:
    """Lattice levels, stencil and workspace layout (host-only)."""
    L = cp_msm_layout()
    lo, hi = domain
    rc = library().cp_msm_layout_of(int(n_atoms), *_grid(shape, origin, h), _vec3(lo), _vec3(hi),
                                    float(np.float32(cutoff)), float(np.float32(lattice_h)), ctypes.byref(L))
    _check(rc, "cp_msm_layout_of")
    return L


def msm_workspace_bytes(n_atoms, shape, origin, h, cutoff, lattice_h, domain) -> int:
    return int(msm_layout(n_atoms, shape, origin, h, cutoff, lattice_h, domain).total_bytes)


def msm_longrange(atoms, shape, origin, h, cutoff, lattice_h, domain=None, accumulate: bool = False,
                  workspace=None, out=None, stream=None, host_out=None):
    """Multilevel approximation of V_long = sum_a q_a g_c(r) (the smooth part
    of 1/r that the cutoff sum leaves out); returns V as (nz, ny, nx).

    ``domain``: ((lo x, y, z), (hi x, y, z)) containing every atom; if None,
    the atoms' bounding box from ``atom_bounds``.  ``accumulate`` adds into
    ``out`` instead of overwriting it."""
    lib = library()
    dev_atoms, on_host = _as_device_atoms(atoms)
    n = int(dev_atoms.shape[0])
    lo, hi = _domain(domain, dev_atoms, stream)
    need = msm_workspace_bytes(n, shape, origin, h, cutoff, lattice_h, (lo, hi))
    ws = _workspace(workspace, need, dev_atoms.device)
    if accumulate and out is None:
        raise ValueError("accumulate=True needs out")
    V = _out_tensor(out, shape, dev_atoms.device)
    rc = lib.cp_msm_longrange(dev_atoms.data_ptr() if n else None, n, *_grid(shape, origin, h), _vec3(lo), _vec3(hi),
                              float(np.float32(cutoff)), float(np.float32(lattice_h)), ws.data_ptr(),
                              ws.numel() * ws.element_size(), V.data_ptr(), int(bool(accumulate)), _stream(stream))
    _check(rc, "cp_msm_longrange")
    return _finish_host(V, host_out) if on_host else V


def msm_map(atoms, shape, origin, h, cutoff, bin_size, lattice_h, capacity: int = 0, domain=None, out=None,
            stream=None, host_out=None):
    """Multilevel approximation of the full direct sum: the cutoff map (short
    range) plus the long-range part, both through the library."""
    dev_atoms, on_host = _as_device_atoms(atoms)
    V = _cutoff_sum(dev_atoms, shape, origin, h, cutoff, bin_size, capacity, out=out, stream=stream)
    msm_longrange(dev_atoms, shape, origin, h, cutoff, lattice_h, domain=domain, accumulate=True, out=V,
                  stream=stream)
    return _finish_host(V, host_out) if on_host else V
