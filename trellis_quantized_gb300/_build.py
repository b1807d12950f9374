"""Build libexl3.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each CUDA translation unit under csrc/ compiles in parallel to an object; the
objects link into ``_build/libexl3.so``.  The instruction-throughput
microbenchmark under ubench/ links into ``_build/libexl3_ubench.so`` (it is
not part of the library).  A build is skipped when its library is newer than
every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libexl3.so")
UBENCH = os.path.join(PKG, "ubench")
UBENCH_LIB = os.path.join(BUILD, "libexl3_ubench.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libexl3")
    return path


def _inputs(srcdir=CSRC):
    return sorted(glob.glob(os.path.join(srcdir, "*.cu"))), sorted(
        glob.glob(os.path.join(srcdir, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib=LIB, srcdir=CSRC) -> bool:
    if not os.path.exists(lib):
        return False
    srcs, hdrs = _inputs(srcdir)
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in srcs + hdrs + [__file__])


def build_ubench(force: bool = False, verbose: bool = False) -> str:
    """The instruction-throughput microbenchmark (bench.py --only pipes)."""
    return build(force, verbose, lib=UBENCH_LIB, srcdir=UBENCH)


def build(force: bool = False, verbose: bool = False, lib: str = LIB, srcdir: str = CSRC) -> str:
    if not force and up_to_date(lib, srcdir):
        return lib
    objdir = os.path.join(BUILD, "obj" if lib == LIB else "obj_" + os.path.basename(srcdir))
    os.makedirs(objdir, exist_ok=True)
    srcs, _ = _inputs(srcdir)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(16, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
    print(build_ubench(force=True, verbose=True))
