"""Exact arithmetic used to pin the oracle; independent of it and of numpy's codec.

Every binary16 value is an integer multiple of 2^-24, so a product of two is a
multiple of 2^-48 and a sum of products is held exactly by a Python integer
scaled by 2^-48.  ``round_rational`` rounds an exact rational to a binary
floating-point format (nearest, ties to even) from the format's parameters
alone.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

# (precision in bits including the hidden one, minimum normal exponent, largest finite)
F16_FORMAT = (11, -14, Fraction(65504))
F32_FORMAT = (24, -126, Fraction((2 ** 24 - 1) * 2 ** 104))


def f16_to_int24(bits: np.ndarray) -> np.ndarray:
    """binary16 bit patterns (finite) -> value * 2^24 as Python ints (object array).

    Written from the format definition, not with any float conversion.
    """
    b = np.asarray(bits, np.uint16).astype(np.int64)
    sign = (b >> 15) & 1
    e = (b >> 10) & 0x1F
    f = b & 0x3FF
    if np.any(e == 31):
        raise ValueError("inf/NaN have no exact integer form")
    sig = np.where(e == 0, f, f + 1024)
    shift = np.where(e == 0, 0, e - 1)  # normal: (1024+f) * 2^(e-25) * 2^24 = sig << (e-1)
    out = np.empty(b.shape, dtype=object)
    flat_out = out.reshape(-1)
    for idx, (s, m, sh) in enumerate(zip(sign.reshape(-1), sig.reshape(-1), shift.reshape(-1))):
        v = int(m) << int(sh)
        flat_out[idx] = -v if s else v
    return out


def exact_gemm_int48(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Exact A @ B scaled by 2^48, as an object array of Python ints."""
    ai = f16_to_int24(a_bits)
    bi = f16_to_int24(b_bits)
    M, K = ai.shape
    K2, N = bi.shape
    assert K == K2
    c = np.empty((M, N), dtype=object)
    for i in range(M):
        row = ai[i]
        for j in range(N):
            s = 0
            col = bi[:, j]
            for k in range(K):
                s += row[k] * col[k]
            c[i, j] = s
    return c


def round_rational(q: Fraction, fmt) -> Fraction | float:
    """Nearest value of the binary format to the exact rational q (ties to even).

    Returns a Fraction, or +-inf (as a float) on overflow.
    """
    p, emin, fmax = fmt
    if q == 0:
        return Fraction(0)
    neg = q < 0
    a = -q if neg else q
    # e = floor(log2(a))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - p + 1)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    # overflow: beyond the largest finite value the rounding goes to inf when
    # a is at or past the midpoint to the next (unrepresentable) step
    if r > fmax:
        return float("-inf") if neg else float("inf")
    return -r if neg else r


def distance_to_tie(q: Fraction, fmt) -> Fraction:
    """|q - nearest rounding tie point| for the format (how close q is to a tie)."""
    p, emin, _ = fmt
    if q == 0:
        return Fraction(1)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - p + 1)
    n = a / ulp
    fl = n.numerator // n.denominator
    d = abs(a - (fl + Fraction(1, 2)) * ulp)
    if fl == 2 ** (p - 1) and e > emin:
        # just above a power of two: the tie below it is on the finer grid
        d = min(d, abs(a - (Fraction(2) ** e - ulp / 4)))
    return d
