"""Build libfp8bq.so in-tree with nvcc for sm_103a.

    python -m fp8_precision_pretraining_amax_b300.build [--force] [--verbose]

The library is one CUDA translation unit (csrc/fp8bq.cu) linked against the
static CUDA runtime, so it loads on machines without a GPU (the driver is only
touched on the first CUDA call).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfp8bq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc_command(out: str = LIB, verbose: bool = False):
    cmd = ["nvcc", *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "static", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
           "-I", INCLUDE, "-I", CSRC, "-o", out, os.path.join(CSRC, "fp8bq.cu")]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    proc = subprocess.run(nvcc_command(tmp, verbose), capture_output=True, text=True)
    if proc.returncode != 0:
        sys.stderr.write(proc.stdout + proc.stderr)
        raise RuntimeError("nvcc failed building libfp8bq.so")
    if verbose:
        sys.stderr.write(proc.stdout + proc.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="--verbose" in sys.argv)
    print(LIB)
