"""Builds the CUDA library ``libmoe_gb300.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked into one shared library
next to this file (CUDA runtime linked statically; the driver is reached through the runtime's
entry-point query, so nothing else is needed at load time). The build is skipped when the library
is newer than every source and header and was built on this machine's architecture.
"""

from __future__ import annotations

import glob
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIBRARY = os.path.join(PKG_DIR, "libmoe_gb300.so")
STAMP = os.path.join(BUILD_DIR, "arch.stamp")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH_FLAGS,
    "-O3",
    "-lineinfo",
    "-std=c++17",
    "-Xcompiler", "-fPIC,-O2",
    "-I", INCLUDE,
    "-I", CSRC,
]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libmoe_gb300.so")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def is_stale() -> bool:
    if not os.path.exists(LIBRARY) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as fh:
        if fh.read().strip() != platform.machine():
            return True
    lib_time = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(p) > lib_time for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library if needed. Returns its path."""
    if not force and not is_stale():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stderr}")
        if ptxas_info or verbose:
            sys.stderr.write(res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(sources()), os.cpu_count() or 1))) as pool:
        objs = list(pool.map(compile_one, sources()))
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    with open(STAMP, "w") as fh:
        fh.write(platform.machine())
    return LIBRARY


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIBRARY)
