"""Builds libcpmap.so (the sm_103a CUDA library behind the C ABI) in-tree.

    python -m direct_coulomb_summation_gb300.build [--checked]

Each .cu file is compiled to an object in parallel with nvcc for
``sm_103a`` only, then linked into ``_build/libcpmap.so``.  A stamp of the
sources and flags decides whether a rebuild is needed.

``checked=True`` builds ``_build/libcpmap_checked.so`` from the same sources
with -DCP_BOUNDS_CHECKS: every runtime-computed index of the kernels'
global and shared-memory accesses is tested, and a violation records
CP_DEVICE_RANGE in the device status word and skips the access.  Setting
CPMAP_CHECKED=1 makes the binding load that library.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcpmap.so")
STAMP = os.path.join(BUILD, "libcpmap.stamp")
LIB_CHECKED = os.path.join(BUILD, "libcpmap_checked.so")
STAMP_CHECKED = os.path.join(BUILD, "libcpmap_checked.stamp")
CHECKED_FLAGS = ["-DCP_BOUNDS_CHECKS"]

SOURCES = ["cp_host.cu", "cp_direct.cu", "cp_cutoff.cu", "cp_msm.cu", "cp_probe.cu", "cp_variants.cu"]
HEADERS = ["cp_device.cuh", "cp_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH,
    "-lineinfo",
    "-O3",
    "-std=c++17",
    "-Xcompiler",
    "-fPIC,-ffp-contract=off,-fvisibility=hidden",
    "-Xptxas",
    "-warn-spills",
]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: cannot build libcpmap.so")


def _digest(extra=()) -> str:
    h = hashlib.sha1()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "cpmap.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


def _paths(checked: bool):
    if checked:
        return LIB_CHECKED, STAMP_CHECKED, os.path.join(BUILD, "obj_checked"), CHECKED_FLAGS
    return LIB, STAMP, os.path.join(BUILD, "obj"), []


def up_to_date(checked: bool = False) -> bool:
    lib, stamp, _, extra = _paths(checked)
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == _digest(extra)


def _compile(nvcc: str, src: str, obj: str, verbose: bool, extra=()) -> str:
    cmd = [nvcc, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile (if needed) and return the path of libcpmap.so (or of the
    checked build, libcpmap_checked.so)."""
    lib, stamp, objdir, extra = _paths(checked)
    if not force and up_to_date(checked):
        return lib
    nvcc = nvcc_path()
    os.makedirs(objdir, exist_ok=True)
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        for name in SOURCES:
            src = os.path.join(CSRC, name)
            obj = os.path.join(objdir, name.replace(".cu", ".o"))
            jobs.append((name, pool.submit(_compile, nvcc, src, obj, verbose, extra)))
        logs = [(name, fut.result()) for name, fut in jobs]
    if verbose:
        for name, log in logs:
            if log.strip():
                print(f"--- {name}\n{log}", file=sys.stderr)
    objs = [os.path.join(objdir, n.replace(".cu", ".o")) for n in SOURCES]
    tmp = lib + f".tmp{os.getpid()}"
    res = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(_digest(extra))
    return lib


def build_all(force: bool = False) -> tuple:
    """Both libraries, compiled concurrently: (release path, checked path)."""
    with cf.ThreadPoolExecutor(max_workers=2) as pool:
        rel = pool.submit(build, force, False, False)
        chk = pool.submit(build, force, False, True)
        return rel.result(), chk.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
