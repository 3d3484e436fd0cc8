"""CPU oracle for the pipelined tiled fp16 GEMM.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library under ``tensor_core_tiled_02_gb300`` and its binding) never does,
and the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 accumulation, its own
binary16 codec); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  What it computes follows "Quickstart: GPU", section
"Pipelining: a matmul kernel": ``matmul(a, b, out_dtype)`` with an fp32
accumulator and ``astype(out_dtype)``, checked against the untiled ``a @ b``.  The oracle is that untiled
product in fp64, rounded once to the output type.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

OUT_F16 = 0
OUT_F32 = 1
OUT_F64 = 2  # the unrounded fp64 sums

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library; return its path.

    ``-ffp-contract=off`` keeps every multiply and add a separate IEEE
    operation on both x86 and Arm (each binary16 x binary16 product is exact
    in binary64, so a fused multiply-add would give the same sums, but the
    flag makes that independent of the argument).
    """
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           *extra_flags, "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    lib.oracle_f16_decode.restype = ctypes.c_double
    lib.oracle_f16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_round.restype = ctypes.c_uint16
    lib.oracle_f16_round.argtypes = [ctypes.c_double]
    lib.oracle_f32_round.restype = ctypes.c_float
    lib.oracle_f32_round.argtypes = [ctypes.c_double]
    lib.oracle_f16_decode_array.restype = None
    lib.oracle_f16_decode_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_f16_round_array.restype = None
    lib.oracle_f16_round_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_gemm_rows.restype = ctypes.c_int
    lib.oracle_gemm_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
    lib.oracle_gemm_rows_decoded.restype = ctypes.c_int
    lib.oracle_gemm_rows_decoded.argtypes = lib.oracle_gemm_rows.argtypes
    lib.oracle_gemm_acc_rows.restype = ctypes.c_int
    lib.oracle_gemm_acc_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
    lib.oracle_add_f32.restype = None
    lib.oracle_add_f32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.oracle_gemm_elems.restype = ctypes.c_int
    lib.oracle_gemm_elems.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    del u16p
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.

    With ``path`` given, load that build instead of the default one (used by
    the tests that check the pins catch a deliberately broken oracle).
    """
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _u16(x) -> np.ndarray:
    """fp16 data as a contiguous uint16 array of its bit patterns."""
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected float16 or uint16 bit patterns, got {x.dtype}")
    return np.ascontiguousarray(x)


def _out_np_dtype(out_dtype: int):
    return {OUT_F16: np.uint16, OUT_F32: np.float32, OUT_F64: np.float64}[out_dtype]


def _threads(nthreads):
    return nthreads if nthreads else (os.cpu_count() or 1)


def decode_f16(bits, lib=None) -> np.ndarray:
    lib = lib or load()
    b = _u16(bits).ravel()
    out = np.empty(b.shape, np.float64)
    lib.oracle_f16_decode_array(b.ctypes.data, out.ctypes.data, b.size)
    return out.reshape(np.shape(bits))


def round_f16(x, lib=None) -> np.ndarray:
    """fp64 -> binary16 bit patterns (uint16), nearest-even."""
    lib = lib or load()
    a = np.ascontiguousarray(np.asarray(x, np.float64)).ravel()
    out = np.empty(a.shape, np.uint16)
    lib.oracle_f16_round_array(a.ctypes.data, out.ctypes.data, a.size)
    return out.reshape(np.shape(x))


def gemm(A, B, out_dtype: int = OUT_F16, rows=None, nthreads=None, lib=None) -> np.ndarray:
    """C_ref = round_out(A @ B) over fp64, for the listed rows (all by default).

    ``A`` is [M, K], ``B`` is [K, N], both float16 (or their uint16 bits).
    Returns a [len(rows), N] array: uint16 bit patterns for OUT_F16, float32
    for OUT_F32, float64 for OUT_F64.
    """
    lib = lib or load()
    a = _u16(A)
    b = _u16(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch {a.shape} @ {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, np.int64)).ravel()
    out = np.zeros((rows.size, N), _out_np_dtype(out_dtype))
    rc = lib.oracle_gemm_rows(a.ctypes.data, b.ctypes.data, out.ctypes.data, M, N, K,
                              out_dtype, rows.ctypes.data, rows.size, _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_rows failed with {rc}")
    return out


def gemm_acc(A, B, Cin, out_dtype: int = OUT_F16, rows=None, nthreads=None, lib=None) -> np.ndarray:
    """round_out(Cin + A @ B) over fp64, the sum starting from Cin, for the
    listed rows.  ``Cin`` is [M, N] float16 (or its uint16 bits) or float32."""
    lib = lib or load()
    a = _u16(A)
    b = _u16(B)
    cin = np.asarray(Cin)
    if cin.dtype == np.float32:
        cin_dtype = OUT_F32
    else:
        cin = _u16(cin)
        cin_dtype = OUT_F16
    cin = np.ascontiguousarray(cin)
    M, K = a.shape
    N = b.shape[1]
    if cin.shape != (M, N):
        raise ValueError(f"Cin must be {(M, N)}, got {cin.shape}")
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, np.int64)).ravel()
    out = np.zeros((rows.size, N), _out_np_dtype(out_dtype))
    rc = lib.oracle_gemm_acc_rows(a.ctypes.data, b.ctypes.data, cin.ctypes.data, cin_dtype, out.ctypes.data, M, N,
                                  K, out_dtype, rows.ctypes.data, rows.size, _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_acc_rows failed with {rc}")
    return out


def add_f32(X, Y, lib=None) -> np.ndarray:
    """Z = X + Y, one binary32 addition per element (the blocked add's result)."""
    lib = lib or load()
    x = np.ascontiguousarray(np.asarray(X, np.float32))
    y = np.ascontiguousarray(np.asarray(Y, np.float32))
    if x.shape != y.shape:
        raise ValueError("X and Y differ in shape")
    z = np.empty_like(x)
    lib.oracle_add_f32(x.ctypes.data, y.ctypes.data, z.ctypes.data, x.size)
    return z


class DecodedB:
    """B decoded once to fp64, for computing many row samples of one product."""

    def __init__(self, B, lib=None):
        self.lib = lib or load()
        b = _u16(B)
        self.K, self.N = b.shape
        self.bd = np.empty(b.shape, np.float64)
        self.lib.oracle_f16_decode_array(b.ctypes.data, self.bd.ctypes.data, b.size)

    def gemm_rows(self, A, rows, out_dtype: int = OUT_F16, nthreads=None) -> np.ndarray:
        a = _u16(A)
        M, K = a.shape
        if K != self.K:
            raise ValueError("inner dimensions differ")
        rows = np.ascontiguousarray(np.asarray(rows, np.int64)).ravel()
        out = np.zeros((rows.size, self.N), _out_np_dtype(out_dtype))
        rc = self.lib.oracle_gemm_rows_decoded(a.ctypes.data, self.bd.ctypes.data, out.ctypes.data, M,
                                               self.N, K, out_dtype, rows.ctypes.data, rows.size,
                                               _threads(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_gemm_rows_decoded failed with {rc}")
        return out


def gemm_elems(A, B, ii, jj, out_dtype: int = OUT_F16, lib=None) -> np.ndarray:
    """C_ref[ii[t], jj[t]] for each t, computed one element at a time."""
    lib = lib or load()
    a = _u16(A)
    b = _u16(B)
    M, K = a.shape
    N = b.shape[1]
    ii = np.ascontiguousarray(np.asarray(ii, np.int64)).ravel()
    jj = np.ascontiguousarray(np.asarray(jj, np.int64)).ravel()
    if ii.shape != jj.shape:
        raise ValueError("index arrays differ in length")
    out = np.zeros(ii.shape, _out_np_dtype(out_dtype))
    rc = lib.oracle_gemm_elems(a.ctypes.data, b.ctypes.data, out.ctypes.data, M, N, K,
                               out_dtype, ii.ctypes.data, jj.ctypes.data, ii.size)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_elems failed with {rc}")
    return out


def as_values(c: np.ndarray, out_dtype: int) -> np.ndarray:
    """Oracle output as float64 values (decoding binary16 bits with numpy)."""
    if out_dtype == OUT_F16:
        return c.view(np.float16).astype(np.float64)
    return c.astype(np.float64)
