"""Build the in-tree C-ABI library ``libnvfp4_gemv.so`` for sm_103a.

Usage: ``python -m nvfp4_weight_quantized_gemv_gb300.buildlib`` (or ``build()``).
Translation units compile in parallel with nvcc, then link into one shared
library next to this file.  Static cudart, one -gencode (compute_103a/sm_103a).
``build(debug_bounds=True)`` makes ``libnvfp4_gemv_debug.so`` from the same
sources with -DNVFP4_DEBUG_BOUNDS: the kernels' computed workspace indices
are checked on the device (a failed check sets a bit of the device error
word and skips the access).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnvfp4_gemv.so")
OBJ_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libnvfp4_gemv_debug.so")
SOURCES = ["gemv_stream.cu", "gemv_tc.cu", "gemv_fp4.cu", "gemv_generic.cu", "abi.cu", "quantize_host.cpp", "gemv_noalloc.cu",
           "quantize_gpu.cu", "moe_gemv.cu", "moe_mma.cu",
           "selftest.cu"]
HEADERS = ["ptx.cuh", "tcgen05.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _flags(src: str, debug_bounds: bool = False):
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-ffp-contract=off",
              "-I", os.path.join(ROOT, "include"), "-I", CSRC] + (["-DNVFP4_DEBUG_BOUNDS"] if debug_bounds else [])
    if src.endswith(".cu"):
        return ARCH + common + ["-Xptxas", "-v"]
    return common


def _newest_input() -> float:
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "nvfp4_gemv.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    lib, objdir = (LIB_DEBUG, OBJ_DEBUG) if debug_bounds else (LIB, OBJ)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    nvcc = nvcc_path()
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc] + _flags(src, debug_bounds) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """The release and the debug-bounds library, compiled side by side."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build, force, False, False), ex.submit(build, force, False, True)]:
            f.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug_bounds="--debug-bounds" in sys.argv))
