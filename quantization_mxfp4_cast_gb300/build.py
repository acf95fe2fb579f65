"""Builds libmxfp4.so (the CUDA kernels + C ABI) in-tree with nvcc for sm_103a.

Each .cu file compiles in parallel to an object, then one nvcc link step makes
the shared library.  The result sits next to this file; nothing is installed.
An object is rebuilt when its source or ANY header under csrc/ or include/ is
newer than it (every translation unit may include every header, directly or
not, so the headers are not tracked per file).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG_DIR), "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libmxfp4.so")
SOURCES = ["cast.cu", "gemm.cu", "api.cu", "noalloc.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def headers(csrc: str = CSRC, include: str = INCLUDE) -> list:
    """Every header a translation unit may include."""
    found = []
    for d in (csrc, include):
        for pat in ("*.h", "*.cuh", "*.hpp"):
            found += glob.glob(os.path.join(d, pat))
    return sorted(found)


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def stale_sources(csrc: str = CSRC, include: str = INCLUDE, build_dir: str = BUILD_DIR,
                  sources=SOURCES, force: bool = False) -> list:
    """The sources whose object must be recompiled."""
    hdrs = headers(csrc, include)
    out = []
    for src in sources:
        s = os.path.join(csrc, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + hdrs):
            out.append(src)
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = [os.path.join(BUILD_DIR, src.replace(".cu", ".o")) for src in SOURCES]
    jobs = [[nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o",
             os.path.join(BUILD_DIR, src.replace(".cu", ".o"))]
            for src in stale_sources(force=force)]

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("nvcc link failed")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
