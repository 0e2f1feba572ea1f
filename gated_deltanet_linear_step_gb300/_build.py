"""Builds the in-tree CUDA library ``libgdn.so`` for sm_103a with nvcc.

The library is compiled from ``csrc/`` (the kernels and the C ABI declared in
``include/gdn.h``); object files go to ``_build/`` next to this file and the
shared library to this package folder. Both are build artefacts, not sources.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
SOURCES = ["gdn_step.cu", "gdn_decode_t1.cu", "gdn_chunk.cu", "gdn_window_tc.cu", "gdn_ab.cu", "gdn_proj.cu", "gdn_proj_noalloc.cu", "gdn_host_pipeline.cpp", "gdn_api.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# A standalone measuring program, not linked into the library: the device's FP32 FMA rate.
FMA_RATE_SRC = "fp32_fma_rate.cu"
FMA_RATE_EXE = os.path.join(BUILD, "fp32_fma_rate")


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libgdn.so")


def build(verbose: bool = False) -> str:
    """Compiles every source in parallel and links ``libgdn.so``; returns its path. Also builds the
    FP32 FMA-rate program (``_build/fp32_fma_rate``) from ``csrc/fp32_fma_rate.cu``."""
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + common + ["-Xptxas", "-v", "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    def compile_fma_rate():
        cmd = [cc] + ARCH + ["-O3", "-std=c++17", "-lineinfo", os.path.join(CSRC, FMA_RATE_SRC), "-o", FMA_RATE_EXE]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {FMA_RATE_SRC}:\n{r.stdout}\n{r.stderr}")

    with ThreadPoolExecutor(len(SOURCES) + 1) as ex:
        fma_rate = ex.submit(compile_fma_rate)
        results = list(ex.map(compile_one, SOURCES))
        fma_rate.result()
    if verbose:
        for _, log in results:
            for line in log.splitlines():
                if "registers" in line or "spill" in line:
                    print(line.strip())
    tmp = LIB + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
