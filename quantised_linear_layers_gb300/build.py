"""Builds libqlinear.so from csrc/ with nvcc for sm_103a, in tree.

Each translation unit is compiled in parallel, then linked as a shared
library next to this file. No CUDA math shortcuts (--use_fast_math is never
passed): the cast depends on correctly rounded division.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqlinear.so")
SOURCES = ["api.cu", "cast.cu", "gemm.cu", "gemm_mx.cu", "gemm_mx2.cu", "gemm_mx_sk.cu", "gemm_pair.cu", "gemm_prom_sk.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found")
    return p


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "--expt-relaxed-constexpr"] + list(extra)


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """Compile the library; returns its path. `variant` (e.g. "bounds" with
    extra_flags=("-DQL_BOUNDS_CHECK",)) builds into its own folder and
    libqlinear_<variant>.so, leaving the product library as it is."""
    build_dir = BUILD + (f"_{variant}" if variant else "")
    lib = LIB.replace(".so", f"_{variant}.so") if variant else LIB
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "qlinear.h"))
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            cmd = [nvcc()] + _flags(extra_flags) + ["-c", s, "-o", o]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, r in ex.map(run, jobs):
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build_bounds_checked(force: bool = False) -> str:
    """The debugging build with every plain global access range-checked
    (QL_BOUNDS_CHECK): libqlinear_bounds.so beside the product library."""
    return build(force=force, extra_flags=("-DQL_BOUNDS_CHECK",), variant="bounds")


if __name__ == "__main__":
    import sys
    if "--bounds" in sys.argv:
        print(build_bounds_checked(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
