"""Builds libmxfp8.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into a shared library
next to this file with the CUDA runtime linked statically (the library loads on a
machine without a GPU; CUDA is only needed when a compute call runs).
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmxfp8.so")
SOURCES = ("api.cu", "quantize.cu", "gemm.cu", "selfcheck.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmxfp8.so")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3",
                   "-I", INCLUDE, "-I", CSRC, *extra]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    cmd = [nvcc(), *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _fresh() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps()


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compiles and links libmxfp8.so if any source is newer than it; returns its path.
    Processes that build at once (the ranks of a multi-GPU launch) take turns under a file
    lock, and a process that finds the library fresh once it holds the lock does not
    rebuild it."""
    if not force and _fresh():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and _fresh():
                return LIB
            with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
                objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
            tmp = f"{LIB}.{os.getpid()}.tmp"
            cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, LIB)
            return LIB
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
