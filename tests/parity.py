"""The parity criterion between the CUDA path and the oracle.

Per element:  |C - C_ref| <= 2e-3 |C_ref| + 1e-2 sqrt(K / 1024),
with C_ref the oracle's rounded output.

That bar is loose for small-valued outputs (for N(0,1)/sqrt(K) inputs, std(C)
is 1/64 while the absolute term at K = 4096 is 0.02), so a second, tight
check rides along, derived from the arithmetic:

  * fp16 output: both sides round a near-identical value to fp16 (the GPU
    from its fp32 sum, the oracle from the exact fp64 sum), so the rms of
    C - C_ref over the elements is about one fp16 half-ulp of the typical
    |C|, i.e. 2^-11 |C| / sqrt(3) ~ 3e-4 |C|; a bound of 2e-3 rms(C_ref)
    catches a lost K-block (one of 64 dropped gives 0.125 rms(C_ref)).
  * fp32 output: only the accumulation errs.  The tensor core adds each
    group of 16 products (one tcgen05.mma K slice) to the fp32 accumulator
    with truncating alignment rather than IEEE round-to-nearest per add, so
    the error may grow linearly in the number of groups, not as sqrt(K).
    Bound: 2 fp32 ulps (2^-22 relative) per group, with a floor of 8 groups:
    rms(C - C_ref) <= 2^-22 (K/16 + 8) rms(C_ref).  At K = 32768 that is
    4.9e-4, still 90 times below the 4.4e-2 a single lost K-block gives.
"""
from __future__ import annotations

import numpy as np


def rms_bound(out_dtype: int, K: int) -> float:
    acc = 2.0 ** -22 * (K / 16.0 + 8.0)
    return 2e-3 + acc if out_dtype == 0 else acc


def tolerance(c_ref: np.ndarray, K: int) -> np.ndarray:
    return 2e-3 * np.abs(c_ref) + 1e-2 * np.sqrt(K / 1024.0)


def check(c_gpu: np.ndarray, c_ref: np.ndarray, K: int, out_dtype: int, what: str = "") -> dict:
    """Assert parity; return diagnostics (max and rms error normalised by rms(C_ref))."""
    c_gpu = np.asarray(c_gpu, np.float64)
    c_ref = np.asarray(c_ref, np.float64)
    assert c_gpu.shape == c_ref.shape, (c_gpu.shape, c_ref.shape)
    if c_ref.size == 0:
        return {"n": 0}
    err = np.abs(c_gpu - c_ref)
    tol = tolerance(c_ref, K)
    bad = np.nonzero(~(err <= tol))
    nbad = bad[0].size
    if nbad:
        first = tuple(int(x[0]) for x in bad)
        raise AssertionError(
            f"{what}: {nbad} of {c_ref.size} elements outside tolerance; first at {first}: "
            f"gpu={c_gpu[first]!r} ref={c_ref[first]!r} tol={tol[first]!r}")
    ref_rms = float(np.sqrt(np.mean(c_ref ** 2)))
    err_rms = float(np.sqrt(np.mean(err ** 2)))
    diag = {"n": int(c_ref.size), "max_abs_err": float(err.max()),
            "rms_err_over_rms_ref": err_rms / ref_rms if ref_rms > 0 else err_rms}
    if ref_rms > 0:
        assert err_rms <= rms_bound(out_dtype, K) * ref_rms, f"{what}: rms error too large: {diag}"
    return diag
