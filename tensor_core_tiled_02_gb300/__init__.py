"""Python binding of the sm_103a pipelined tiled fp16 GEMM.

Argument marshalling only: every step of the product runs in the CUDA
library ``libtcgemm.so`` (built in-tree from ``csrc/`` by ``build.py``),
reached through its C ABI (``include/gemm_f16.h``).  PyTorch supplies device
memory and the current stream.  There is no fallback: if the library is
missing the calls raise.

Names follow the C ABI: ``gemm_f16`` (raw pointers), ``gemm_f16_plan``,
``gemm_f16_set_config``, ``gemm_f16_strerror``, ``gemm_f16_device_status``;
``matmul(a, b, out_dtype)`` is the tensor-level call of the ``matmul(a, b,
out_dtype)`` of "Quickstart: GPU", section "Pipelining: a matmul kernel".
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# TCGEMM_VARIANT=trace or =check selects a debug build of the same library
# (libtcgemm_trace.so, libtcgemm_check.so; see build.py); unset: the product
_VARIANT = os.environ.get("TCGEMM_VARIANT", "")
LIB_PATH = os.path.join(_HERE, f"libtcgemm_{_VARIANT}.so" if _VARIANT else "libtcgemm.so")

GEMM_OUT_F16 = 0
GEMM_OUT_F32 = 1

STATUS = {
    0: "GEMM_OK", -1: "GEMM_ERR_NULL", -2: "GEMM_ERR_DIM", -3: "GEMM_ERR_DTYPE",
    -4: "GEMM_ERR_ALIGN", -5: "GEMM_ERR_ALIAS", -6: "GEMM_ERR_CONFIG", -7: "GEMM_ERR_TMAP",
    -8: "GEMM_ERR_LAUNCH", -9: "GEMM_ERR_CUDA", -10: "GEMM_ERR_ARCH", -11: "GEMM_ERR_DEVICE_TIMEOUT",
    -12: "GEMM_ERR_WORKSPACE", -13: "GEMM_ERR_SCRATCH_LIMIT",
}
EXPORTED = ["add_matrices_f32", "gemm_f16", "gemm_f16_acc", "gemm_f16_ws", "gemm_f16_noalloc", "gemm_f16_workspace_size", "gemm_f16_plan",
            "gemm_f16_plan_ws",
            "gemm_f16_set_config", "gemm_f16_get_config", "gemm_f16_strerror", "gemm_f16_device_status",
            "gemm_f16_abi_version"]


class GemmPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "cta_group", "tile_m", "tile_n", "tile_k", "tiles_m", "tiles_n", "num_tiles", "k_steps", "stages",
        "release", "slots", "split", "grid", "raster_group", "smem_bytes", "tmem_cols", "threads",
        "dp_tiles", "sk_tiles", "sk_pairs")] + [("workspace_bytes", ctypes.c_longlong)] + [
        (n, ctypes.c_int) for n in ("sk_split", "sk_helper_tiles")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class GemmConfig(ctypes.Structure):
    _fields_ = [("tile_n", ctypes.c_int), ("stages", ctypes.c_int), ("release", ctypes.c_int),
                ("grid", ctypes.c_int), ("raster_group", ctypes.c_int),
                ("wait_limit", ctypes.c_longlong), ("split", ctypes.c_int), ("cta_group", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("stream_k", ctypes.c_int), ("inject_stall", ctypes.c_int)]


class GemmError(RuntimeError):
    def __init__(self, code: int, where: str = "gemm_f16"):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({strerror(code)})")


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m tensor_core_tiled_02_gb300.build` "
                    "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            vp, ci = ctypes.c_void_p, ctypes.c_int
            lib.gemm_f16.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
            lib.gemm_f16.restype = ci
            lib.gemm_f16_plan.argtypes = [ci, ci, ci, ci, ci, ctypes.POINTER(GemmPlan)]
            lib.gemm_f16_plan.restype = ci
            lib.gemm_f16_plan_ws.argtypes = [ci, ci, ci, ci, ci, ctypes.POINTER(GemmPlan)]
            lib.gemm_f16_plan_ws.restype = ci
            lib.gemm_f16_ws.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp, ctypes.c_size_t, vp]
            lib.gemm_f16_ws.restype = ci
            lib.add_matrices_f32.argtypes = [vp, vp, vp, ci, ci, vp]
            lib.add_matrices_f32.restype = ci
            lib.gemm_f16_acc.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
            lib.gemm_f16_acc.restype = ci
            lib.gemm_f16_noalloc.argtypes = [vp, vp, vp, ci, ci, ci, ci, vp]
            lib.gemm_f16_noalloc.restype = ci
            lib.gemm_f16_workspace_size.argtypes = [ci, ci, ci, ci, ci, ctypes.POINTER(ctypes.c_size_t)]
            lib.gemm_f16_workspace_size.restype = ci
            lib.gemm_f16_set_config.argtypes = [ctypes.POINTER(GemmConfig)]
            lib.gemm_f16_set_config.restype = ci
            lib.gemm_f16_get_config.argtypes = [ctypes.POINTER(GemmConfig)]
            lib.gemm_f16_get_config.restype = ci
            lib.gemm_f16_strerror.argtypes = [ci]
            lib.gemm_f16_strerror.restype = ctypes.c_char_p
            lib.gemm_f16_device_status.argtypes = [ctypes.POINTER(ci), ci]
            lib.gemm_f16_device_status.restype = ci
            lib.gemm_f16_abi_version.argtypes = []
            lib.gemm_f16_abi_version.restype = ci
            _lib = lib
        return _lib


def strerror(code: int) -> str:
    return load_library().gemm_f16_strerror(int(code)).decode()


def gemm_f16(A: int, B: int, C: int, M: int, N: int, K: int, out_dtype: int, stream: int = 0) -> int:
    """The C entry point on raw device pointers (ints); returns its status code."""
    return load_library().gemm_f16(A, B, C, M, N, K, out_dtype, stream)


def gemm_f16_ws(A: int, B: int, C: int, M: int, N: int, K: int, out_dtype: int, workspace: int,
                workspace_bytes: int, stream: int = 0) -> int:
    """The C entry point with a stream-K workspace (raw device pointers); returns its status."""
    return load_library().gemm_f16_ws(A, B, C, M, N, K, out_dtype, workspace, workspace_bytes, stream)


def gemm_f16_plan(M: int, N: int, K: int, out_dtype: int = GEMM_OUT_F16, num_sms: int = 0,
                  with_workspace: bool = False) -> dict:
    p = GemmPlan()
    fn = load_library().gemm_f16_plan_ws if with_workspace else load_library().gemm_f16_plan
    rc = fn(M, N, K, out_dtype, num_sms, ctypes.byref(p))
    if rc != 0:
        raise GemmError(rc, "gemm_f16_plan")
    return p.as_dict()


def gemm_f16_workspace_size(M: int, N: int, K: int, out_dtype: int = GEMM_OUT_F16, num_sms: int = 0) -> int:
    n = ctypes.c_size_t(0)
    rc = load_library().gemm_f16_workspace_size(M, N, K, out_dtype, num_sms, ctypes.byref(n))
    if rc != 0:
        raise GemmError(rc, "gemm_f16_workspace_size")
    return n.value


def workspace(M: int, N: int, K: int, out_dtype=GEMM_OUT_F16, device=None):
    """A zero-filled device workspace for gemm_f16_ws / matmul(workspace=...),
    or None when the problem's plan needs none (torch allocates it)."""
    import torch

    nbytes = gemm_f16_workspace_size(M, N, K, _out_code(out_dtype))
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device if device is not None else "cuda")


def gemm_f16_set_config(**fields) -> None:
    """Set the tuning override; no arguments restores the defaults."""
    cfg = GemmConfig()
    for k, v in fields.items():
        if not hasattr(cfg, k):
            raise TypeError(f"unknown config field {k!r}")
        setattr(cfg, k, int(v))
    rc = load_library().gemm_f16_set_config(ctypes.byref(cfg) if fields else None)
    if rc != 0:
        raise GemmError(rc, "gemm_f16_set_config")


def gemm_f16_get_config() -> dict:
    cfg = GemmConfig()
    rc = load_library().gemm_f16_get_config(ctypes.byref(cfg))
    if rc != 0:
        raise GemmError(rc, "gemm_f16_get_config")
    return {n: getattr(cfg, n) for n, _ in cfg._fields_}


def gemm_f16_device_status(reset: bool = True):
    """(status code, wait site) after synchronising the current device."""
    site = ctypes.c_int(0)
    rc = load_library().gemm_f16_device_status(ctypes.byref(site), int(bool(reset)))
    return rc, site.value


def _check_device(*tensors) -> None:
    """Every tensor handed to the library must live on one CUDA device: the
    kernels take raw device pointers, and a host or another GPU's pointer
    there is a user error caught here, not in a kernel."""
    dev = None
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("every tensor must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices: {dev} and {t.device}")


def _out_code(out_dtype) -> int:
    import torch

    if out_dtype in (torch.float16, GEMM_OUT_F16):
        return GEMM_OUT_F16
    if out_dtype in (torch.float32, GEMM_OUT_F32):
        return GEMM_OUT_F32
    raise ValueError(f"out_dtype must be torch.float16 or torch.float32, got {out_dtype}")


def add_matrices(x, y, out=None, stream=None):
    """Z = x + y for f32 CUDA tensors [M, N] (the pipelined blocked add); ``out``
    may be x or y (in place).  Asynchronous on ``stream``."""
    import torch

    if x.dtype != torch.float32 or y.dtype != torch.float32 or x.shape != y.shape or x.dim() != 2:
        raise ValueError("x and y must be f32 tensors of one 2-D shape")
    if not (x.is_cuda and y.is_cuda and x.is_contiguous() and y.is_contiguous()):
        raise ValueError("x and y must be contiguous CUDA tensors")
    if out is None:
        out = torch.empty_like(x)
    elif out.dtype != torch.float32 or out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous f32 tensor of x's shape")
    _check_device(x, y, out)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(x.device):
        rc = load_library().add_matrices_f32(x.data_ptr(), y.data_ptr(), out.data_ptr(), x.shape[0], x.shape[1],
                                             handle)
    if rc != 0:
        raise GemmError(rc, "add_matrices_f32")
    return out


def matmul_acc(a, b, c, stream=None):
    """c += a @ b in place (c fp16 or fp32, [M, N], contiguous); returns c.

    The library reads c's values before the call and adds the product to them
    in fp32, rounding once to c's type.  Asynchronous on ``stream``.
    """
    import torch

    if a.dtype != torch.float16 or b.dtype != torch.float16:
        raise ValueError("a and b must be torch.float16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch: {tuple(a.shape)} @ {tuple(b.shape)}")
    if c.dtype not in (torch.float16, torch.float32) or tuple(c.shape) != (a.shape[0], b.shape[1]):
        raise ValueError("c must be an fp16 or fp32 [M, N] tensor")
    if not (a.is_contiguous() and b.is_contiguous() and c.is_contiguous()):
        raise ValueError("a, b and c must be contiguous row-major")
    _check_device(a, b, c)
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    code = GEMM_OUT_F16 if c.dtype == torch.float16 else GEMM_OUT_F32
    with torch.cuda.device(a.device):
        rc = load_library().gemm_f16_acc(a.data_ptr(), b.data_ptr(), c.data_ptr(), a.shape[0], b.shape[1],
                                         a.shape[1], code, handle)
    if rc != 0:
        raise GemmError(rc, "gemm_f16_acc")
    return c


def matmul(a, b, out_dtype=None, out=None, stream=None, workspace=None):
    """C = a @ b for fp16 CUDA tensors a [M, K] and b [K, N]; C is fp16 (default) or fp32.

    The kernel is enqueued on ``stream`` (default: torch's current stream) and
    the call returns without synchronising.  ``workspace``: a CUDA tensor from
    ``workspace(...)`` (zero-filled before its first use) enables stream-K.
    Raises ``GemmError`` on a nonzero status from the library and
    ``ValueError`` on tensors it cannot take.
    """
    import torch

    if out_dtype is None:
        out_dtype = torch.float16
    code = _out_code(out_dtype)
    tdt = torch.float16 if code == GEMM_OUT_F16 else torch.float32
    if a.dtype != torch.float16 or b.dtype != torch.float16:
        raise ValueError("a and b must be torch.float16")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch: {tuple(a.shape)} @ {tuple(b.shape)}")
    if not (a.is_cuda and b.is_cuda):
        raise ValueError("a and b must be CUDA tensors")
    if not (a.is_contiguous() and b.is_contiguous()):
        raise ValueError("a and b must be contiguous row-major")
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=tdt, device=a.device)
    elif out.dtype != tdt or tuple(out.shape) != (M, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] tensor of out_dtype")
    _check_device(a, b, out, *([workspace] if workspace is not None else []))
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(a.device):
        if workspace is None:
            rc = gemm_f16(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, code, handle)
        else:
            rc = gemm_f16_ws(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, code, workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), handle)
    if rc != 0:
        raise GemmError(rc)
    return out
