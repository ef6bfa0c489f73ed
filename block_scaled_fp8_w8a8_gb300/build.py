"""Build the CUDA library (sm_103a) in-tree: block_scaled_fp8_w8a8_gb300/_build/.

Each translation unit is compiled by its own nvcc process, in parallel, then
linked into one shared library with the C ABI of include/w8a8_block_fp8.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB_NAME = "libw8a8_gb300.so"
# The debug-bounds build (every kernel checks its global-memory and TMA indexes
# and records W8A8_ERR_DEVICE_BOUNDS instead of an access outside a buffer).
OUT_DEBUG = os.path.join(HERE, "_build_debug")
LIB_NAME_DEBUG = "libw8a8_gb300_debug.so"
UNITS = ["api.cu", "status.cu", "gemm_tiled.cu", "gemm_swapab.cu", "noalloc.cu", "quant.cu", "hostio.cu",
         "gemm_smallm.cu", "gemm_pair.cu", "gemm_generic.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
HEADERS = ["ptx.cuh", "kernels.cuh", "epilogue.cuh", "promote.cuh", "dispatch_table.h", "tuning_table.inc"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def lib_path(debug_bounds: bool = False) -> str:
    return os.path.join(OUT_DEBUG, LIB_NAME_DEBUG) if debug_bounds else os.path.join(OUT, LIB_NAME)


def _flags(verbose: bool, debug_bounds: bool = False):
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                "-I", os.path.join(HERE, "..", "include")]
    if debug_bounds:
        f += ["-DW8A8_DEBUG_BOUNDS=1"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(SRC, h) for h in HEADERS] + \
        [os.path.join(HERE, "..", "include", "w8a8_block_fp8.h")]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link the library; debug_bounds=True builds the debug-bounds
    library (its own objects and .so) instead of the release one."""
    out = OUT_DEBUG if debug_bounds else OUT
    os.makedirs(out, exist_ok=True)
    cc = nvcc()

    def compile_unit(u):
        src = os.path.join(SRC, u)
        obj = os.path.join(out, u.replace(".cu", ".o"))
        if not force and not _stale(obj, src):
            return obj, ""
        cmd = [cc] + _flags(verbose, debug_bounds) + ["-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {u}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_unit, UNITS))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            if log:
                print(log)
    lib = lib_path(debug_bounds)
    if force or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
