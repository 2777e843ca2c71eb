"""Build the CUDA library in-tree: dense_fp16_tensor_tma_gb300/_build/libgemm_f16.so.

Two translation units (the GEMM entry points and the attention forward),
compiled in parallel for sm_103a only and linked into one shared library.
The CUDA runtime is linked statically, so the library needs nothing at load
time beyond libc/libstdc++ (the driver is reached through the runtime when a
call runs).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libgemm_f16.so")
SOURCES = ["gemm_f16.cu", "attn_f16.cu"]
DEPS = ["gemm_f16.cu", "gemm_kernels.cuh", "gemm_kernels_pair.cuh", "gemm_kernels_swap.cuh", "ptx.cuh",
        "attn_f16.cu", "attn_kernels.cuh"]
HEADERS = ["gemm_f16.h", "attn_f16.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(INCLUDE, h) for h in HEADERS]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:   # compile the translation units in parallel
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + tag + ".o")   # nvcc goes by the extension
        cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
        procs.append((subprocess.Popen(cmd), cmd))
        objs.append(obj)
    failed = [cmd for proc, cmd in procs if proc.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    tmp = LIB + tag
    subprocess.check_call([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    for obj in objs:
        os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
