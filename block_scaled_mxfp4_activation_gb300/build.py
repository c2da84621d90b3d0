"""Builds libmxfp4.so in-tree (``block_scaled_mxfp4_activation_gb300/_build/``)
with nvcc for sm_103a.  The translation units compile in parallel; the
library links the CUDA runtime statically and finds the driver's tensor-map
encoder at run time, so it needs no libcuda at link time.

``build(checked=True)`` makes libmxfp4_checked.so from the same sources with
-DMXFP4_CHECKED: every computed-index global or shared-memory access the
kernels make outside a TMA copy is tested against its buffer first, and one
that falls outside is skipped and reported in the device error word (bit 8).
It exists for tests; the normal library compiles those tests away."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmxfp4.so")
CHECKED_LIB = os.path.join(BUILD, "libmxfp4_checked.so")
SOURCES = ["api.cu", "gemm.cu", "chain.cu", "quantize.cu", "no_alloc.cu", "host_copy.cu"]
HEADERS = ["internal.h", "ptx.cuh", "quant.cuh", "tile.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--ptxas-options=-v", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(ROOT, "include", "mxfp4.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile (if stale) and return the path of libmxfp4.so, or of
    libmxfp4_checked.so with `checked`."""
    lib = CHECKED_LIB if checked else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    defines = ["-DMXFP4_CHECKED"] if checked else []

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *[o for o, _ in results], "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
