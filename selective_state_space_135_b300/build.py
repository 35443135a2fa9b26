"""Build the sm_103a CUDA library in-tree (nvcc, no JIT cache).

    python -m selective_state_space_135_b300.build [--force] [-v]

Every .cu file under csrc/ is compiled to an object, then the objects are
linked into libmamba_scan.so.  The same sources are also compiled with
-DMAMBA_DEBUG into libmamba_scan_debug.so, whose kernels check the index of
every global access (see mamba_debug_build in include/mamba_scan.h).  All
objects of both libraries compile in parallel.
"""

from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SRCS = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
DEPS = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(ROOT, "include", "mamba_scan.h")]
LIB = os.path.join(HERE, "libmamba_scan.so")
LIB_DEBUG = os.path.join(HERE, "libmamba_scan_debug.so")
OBJ_DIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in (*SRCS, *DEPS, __file__))


def build(force: bool = False, verbose: bool = False) -> str:
    """Build both libraries if a source is newer; returns the release path."""
    variants = [(lib, extra) for lib, extra in ((LIB, []), (LIB_DEBUG, ["-DMAMBA_DEBUG"]))
                if force or not up_to_date(lib)]
    if not variants:
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    base = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include")]
    if verbose:
        base.insert(0, "-Xptxas=-v")
    jobs = []   # (lib, objs, procs)
    for lib, extra in variants:
        objs, procs = [], []
        for src in SRCS:
            obj = os.path.join(OBJ_DIR, os.path.basename(lib) + "." + os.path.basename(src) + tag + ".o")
            objs.append(obj)
            procs.append(subprocess.Popen([nvcc(), *base, *extra, "-c", "-o", obj, src]))
        jobs.append((lib, objs, procs))
    failed = [src for _, _, procs in jobs for src, p in zip(SRCS, procs) if p.wait() != 0]
    if failed:
        for _, objs, _ in jobs:
            for obj in objs:
                if os.path.exists(obj):
                    os.remove(obj)
        raise RuntimeError(f"nvcc failed on {failed}")
    for lib, objs, _ in jobs:
        tmp = lib + tag
        try:
            subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        finally:
            for obj in objs:
                os.remove(obj)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
