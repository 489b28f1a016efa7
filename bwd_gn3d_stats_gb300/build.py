"""Build step for libgn3d: sm_103a only, output in-tree.

    python -m bwd_gn3d_stats_gb300.build          # builds _build/libgn3d.so and _build/libgn3d_testing.so

Two libraries from the same sources, compiled in parallel: libgn3d.so, the
shipped library (the GroupNorm entry points, diagnostics and nothing else), and
libgn3d_testing.so, compiled with GN3D_TESTING, which adds the testing and
tuning hooks (gn3d_debug_set: launch form, poll budget, forced timeouts, fault
injection, ring sizes; gn3d_debug_get) that the tests use.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgn3d.so")
TESTING_LIB = os.path.join(BUILD, "libgn3d_testing.so")
SOURCES = [os.path.join(CSRC, "gn3d.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
    os.path.join(ROOT, "include", "gn3d.h")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: libgn3d needs the CUDA toolkit to build")


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in DEPS if os.path.exists(d))


def _command(out: str, testing: bool, verbose: bool):
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
           "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-Xlinker", "-rpath," + cuda_lib_dir(), "-o", out] + SOURCES
    if testing:
        cmd.insert(1, "-DGN3D_TESTING")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False) -> str:
    """Build both libraries (the ones out of date); returns the shipped one's path."""
    os.makedirs(BUILD, exist_ok=True)
    jobs = []
    for lib, testing in ((LIB, False), (TESTING_LIB, True)):
        if force or not up_to_date(lib):
            tmp = lib + f".tmp{os.getpid()}"
            jobs.append((subprocess.Popen(_command(tmp, testing, verbose)), tmp, lib))
    failed = None
    for proc, tmp, lib in jobs:
        if proc.wait() != 0:
            failed = lib
        elif failed is None:
            os.replace(tmp, lib)
    if failed:
        raise subprocess.CalledProcessError(1, f"nvcc ({os.path.basename(failed)})")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
