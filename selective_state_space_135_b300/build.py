"""Build the sm_103a CUDA library in-tree (nvcc, no JIT cache).

    python -m selective_state_space_135_b300.build [--force] [-v]

Every .cu file under csrc/ is compiled to an object in parallel, then the
objects are linked into libmamba_scan.so.
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
OBJ_DIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in (*SRCS, *DEPS, __file__))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
             "-I", os.path.join(ROOT, "include")]
    if verbose:
        flags.insert(0, "-Xptxas=-v")
    procs, objs = [], []
    for src in SRCS:
        obj = os.path.join(OBJ_DIR, os.path.basename(src) + tag + ".o")
        objs.append(obj)
        procs.append(subprocess.Popen([nvcc(), *flags, "-c", "-o", obj, src]))
    failed = [src for src, p in zip(SRCS, procs) if p.wait() != 0]
    if failed:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = LIB + tag
    try:
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    finally:
        for obj in objs:
            os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
