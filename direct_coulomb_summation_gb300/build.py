"""Builds libcpmap.so (the sm_103a CUDA library behind the C ABI) in-tree.

    python -m direct_coulomb_summation_gb300.build

Each .cu file is compiled to an object in parallel with nvcc for
``sm_103a`` only, then linked into ``_build/libcpmap.so``.  A stamp of the
sources and flags decides whether a rebuild is needed.
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


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == _digest()


def _compile(nvcc: str, src: str, obj: str, verbose: bool) -> str:
    cmd = [nvcc, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libcpmap.so."""
    if not force and up_to_date():
        return LIB
    nvcc = nvcc_path()
    objdir = os.path.join(BUILD, "obj")
    os.makedirs(objdir, exist_ok=True)
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        for name in SOURCES:
            src = os.path.join(CSRC, name)
            obj = os.path.join(objdir, name.replace(".cu", ".o"))
            jobs.append((name, pool.submit(_compile, nvcc, src, obj, verbose)))
        logs = [(name, fut.result()) for name, fut in jobs]
    if verbose:
        for name, log in logs:
            if log.strip():
                print(f"--- {name}\n{log}", file=sys.stderr)
    objs = [os.path.join(objdir, n.replace(".cu", ".o")) for n in SOURCES]
    tmp = LIB + f".tmp{os.getpid()}"
    res = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_digest())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
