"""Build libawq.so (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: python -m post_bit_weight_awq_b300.build [--force] [--verbose] [--checked]

The library links the CUDA runtime statically, so it loads on a machine with
no GPU (symbol checks) and needs only the driver at run time. --checked builds
libawq_checked.so instead: the same sources with AWQ_CHECKED defined, which
puts a bounds check in front of the kernels' global-memory accesses (a failed
check is counted and the access skipped; awq_bounds_report reads the count).
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libawq.so")
BUILD_DIR = os.path.join(PKG, "_build")
CHECKED_LIB = os.path.join(PKG, "libawq_checked.so")
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3",
    "-std=c++17",
    "-lineinfo",
    "-Xcompiler",
    "-fPIC",
    "-Xcompiler",
    "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in sources() + headers() + [__file__])


def build(force: bool = False, verbose: bool = False, extra=None, checked: bool = False) -> str:
    lib = CHECKED_LIB if checked else LIB
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    objs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        if checked:
            cmd[1:1] = ["-DAWQ_CHECKED"]
        if extra:
            cmd[1:1] = list(extra)
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        objs.append(obj)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers/spills per kernel")
    ap.add_argument("--checked", action="store_true", help="build libawq_checked.so (bounds-checked kernels)")
    a = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if a.ptxas_info else None
    path = build(force=a.force or a.ptxas_info, verbose=a.verbose, extra=extra, checked=a.checked)
    print(path)


if __name__ == "__main__":
    sys.exit(main())
