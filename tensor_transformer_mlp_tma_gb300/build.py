"""Builds libtpmlp.so in-tree: every ``csrc/*.cu`` compiled for sm_103a in parallel
with nvcc, then linked into one shared library next to this file.

A second library, libtpmlp_debug.so, is built from the same sources with
TPMLP_DEBUG=1: the tensor-core GEMM then checks tile coordinates, k-block ranges,
shared-memory addresses and TMEM columns before every access and reports a
failed check in the device status word (TPMLP_ERR_DEVICE) instead of making the
access.  The binding loads it when TPMLP_LIBRARY=debug."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libtpmlp.so")
LIB_DEBUG = os.path.join(HERE, "libtpmlp_debug.so")
BUILD_DIR = os.path.join(ROOT, "_build")
VARIANTS = {LIB: [], LIB_DEBUG: ["-DTPMLP_DEBUG=1"]}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtpmlp.so")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(INCLUDE, "tpmlp.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose_ptxas: bool, defines=(), tag: str = "") -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + tag + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(defines) + (["-Xptxas", "-v"] if verbose_ptxas else []) + \
        ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link libtpmlp.so and libtpmlp_debug.so, each unless it is
    newer than every source; all translation units of both compile in parallel."""
    todo = [lib for lib in VARIANTS if force or not up_to_date(lib)]
    if not todo:
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = sources()
    jobs = [(lib, src) for lib in todo for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[1], verbose_ptxas and j[0] == LIB, VARIANTS[j[0]],
                                              "" if j[0] == LIB else ".debug"), jobs))
    for lib in todo:
        mine = [o for (l2, _), o in zip(jobs, objs) if l2 == lib]
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + mine
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
