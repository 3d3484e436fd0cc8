"""Build the CUDA library in-tree: tensor_core_tiled_02_gb300/libtcgemm.so.

nvcc compiles the kernels for sm_103a only (``-gencode
arch=compute_103a,code=sm_103a``) with the CUDA runtime linked statically, so
the library loads without a GPU and needs no libcuda at link time (the one
driver entry point it uses is fetched at run time).
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
LIB = os.path.join(PKG, "libtcgemm.so")
SOURCES = [os.path.join(CSRC, "gemm_f16.cu")]
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build(verbose_ptxas: bool = False, out: str = LIB, extra=()) -> str:
    cmd = [nvcc_path(), "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, "-I", CSRC,
           "-o", out, *SOURCES, *extra]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)
    return out


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    deps = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(d) > lib_t for d in deps)


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv)
    print(LIB)
