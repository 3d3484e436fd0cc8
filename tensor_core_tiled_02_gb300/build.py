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

# Debug variants of the same sources, each its own library beside the product:
#   trace  -DTCGEMM_TRACE: the kernels stamp %globaltimer and the SM clock per
#          role, tile and K step into a buffer the caller hands the library
#          (gemm_f16_trace_buffer, include/gemm_f16_trace.h); read by trace.py
#   check  -DTCGEMM_CHECK: every shared-memory ring, staging and barrier
#          address and every Tensor Memory column range is checked against
#          its allocation before use; a violation skips the access and is
#          reported through gemm_f16_device_status (sites 9 and 10)
VARIANTS = {"trace": ["-DTCGEMM_TRACE"], "check": ["-DTCGEMM_CHECK"]}


def variant_lib(name: str) -> str:
    return LIB if not name else os.path.join(PKG, f"libtcgemm_{name}.so")


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build(verbose_ptxas: bool = False, out: str | None = None, extra=(), variant: str = "") -> str:
    if variant and variant not in VARIANTS:
        raise ValueError(f"unknown variant {variant!r}")
    out = out or variant_lib(variant)
    cmd = [nvcc_path(), "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, "-I", CSRC,
           *(VARIANTS[variant] if variant else []), "-o", out, *SOURCES, *extra]
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
    v = next((a for a in sys.argv[1:] if a in VARIANTS), "")
    print(build(verbose_ptxas="-v" in sys.argv, variant=v))
