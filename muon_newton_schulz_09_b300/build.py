"""Builds the CUDA library in-tree: muon_newton_schulz_09_b300/lib/libmuon.so.

nvcc cross-compiles for sm_103a on any host; no GPU is needed to build.
Run as ``python -m muon_newton_schulz_09_b300.build`` or call ``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmuon.so")
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(CSRC, "muon_api.cu"), os.path.join(CSRC, "muon_noalloc.cu"),
           os.path.join(CSRC, "muon_shard.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "ns_gemm.cuh", "elementwise.cuh")] + [
    os.path.join(ROOT, "include", "muon.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def cuda_lib_dir() -> str:
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    return os.path.join(home, "lib64")


def command(out: str = LIB, extra=()) -> list:
    return [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC,-O3",
            "-cudart", "shared", "-Xlinker", f"-rpath,{cuda_lib_dir()}", *extra, "-o", out, *SOURCES]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles libmuon.so for sm_103a if any source is newer than it. Returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    tmp = LIB + ".tmp"
    cmd = command(tmp, ("-Xptxas", "-v") if verbose else ())
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
