"""Build the fconv shared library in-tree for sm_103a with nvcc.

    python -m quantized_conv2d_gb300.build [--force] [--verbose]

Produces quantized_conv2d_gb300/libfconv.so (C ABI declared in
include/fconv.h).  The translation units compile in parallel.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfconv.so")
SOURCES = ["fconv_kernels.cu", "fconv_api.cu", "fconv_no_alloc.cu"]
HEADERS = ["fconv_device.cuh", "fconv_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "fconv.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    # host arithmetic (the batch-norm fold) rounds every operation on x86
    # and on Arm alike: no fused multiply-adds from the host compiler; on the
    # device no multiply and add is contracted either (-fmad=false; the
    # epilogue also writes its steps with explicit round-to-nearest
    # intrinsics, each rounded once, in a fixed order)
    common = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-fmad=false",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if verbose:
        common += ["-Xptxas", "-v"]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        procs.append(subprocess.Popen(common + ["-c", os.path.join(CSRC, src), "-o", obj]))
    failed = [p.wait() for p in procs]
    if any(failed):
        raise RuntimeError(f"nvcc failed: {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
    sys.exit(0)
