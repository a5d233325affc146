"""Build libpalu.so (hand-written CUDA for sm_103a) in-tree with nvcc.

Each translation unit is compiled in parallel, then linked into a shared
library next to this file.  No CMake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libpalu.so")
BUILD = os.path.join(HERE, "_build")
# the bounds-checking build (-DPALU_DEBUG_BOUNDS=1): kernels check the block
# indices of their streaming accesses and report PALU_DEVERR_BOUNDS
LIB_DEBUG = os.path.join(HERE, "libpalu_debug.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpalu")
    return exe


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose: bool = False, ptxas_info: bool = False, debug_bounds: bool = False) -> str:
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug_bounds:
        extra.append("-DPALU_DEBUG_BOUNDS=1")

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose or ptxas_info:
        for obj, err in results:
            if err.strip():
                sys.stderr.write(err)
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart_static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
