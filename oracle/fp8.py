"""8-bit floating-point inputs in fp64 -- TEST INFRASTRUCTURE ONLY.

"Kernel 性能从何而来", section "优化 Memory-Bound Kernel": besides tiling,
narrower data types (fp16, fp8, fp4) cut the bytes moved per FLOP.  The FP8
GEMM is the plain GEMM on the values the bytes encode:

    C = alpha * dec(A) * dec(B) + beta * C0

with dec() the exact value of each byte under its format (the two OCP 8-bit
floating-point formats):

  E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
        subnormal (m/8 * 2^-6); no infinities; S.1111.111 is NaN; the largest
        finite magnitude is 1.75 * 2^8 = 448.
  E5M2: sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent 0 is
        subnormal (m/4 * 2^-14); exponent 31 is infinity (m = 0) or NaN; the
        largest finite magnitude is 1.75 * 2^15 = 57344.

Every FP8 value is exact in fp64, so the oracle GEMM on dec(A), dec(B) is
the exact product up to its own fp64 rounding.
"""
from __future__ import annotations

import math

import numpy as np

from . import gemm, to_f64

E4M3, E5M2 = 0, 1
_LAYOUT = {E4M3: (4, 3, 7), E5M2: (5, 2, 15)}   # exponent bits, mantissa bits, bias


def decode_byte(b: int, fmt: int) -> float:
    """Value of one byte under `fmt`, from the field definitions."""
    eb, mb, bias = _LAYOUT[fmt]
    sign = -1.0 if (b >> 7) & 1 else 1.0
    e = (b >> mb) & ((1 << eb) - 1)
    m = b & ((1 << mb) - 1)
    emax = (1 << eb) - 1
    if fmt == E4M3 and e == emax and m == (1 << mb) - 1:
        return math.nan
    if fmt == E5M2 and e == emax:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * (m / (1 << mb)) * 2.0 ** (1 - bias)
    return sign * (1.0 + m / (1 << mb)) * 2.0 ** (e - bias)


def table(fmt: int) -> np.ndarray:
    """fp64 value of every byte 0..255."""
    return np.array([decode_byte(b, fmt) for b in range(256)], dtype=np.float64)


_TABLES = {}


def decode(x, fmt: int) -> np.ndarray:
    """fp64 values of an array of FP8 bytes (uint8 numpy array or torch tensor)."""
    if fmt not in _TABLES:
        _TABLES[fmt] = table(fmt)
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return _TABLES[fmt][np.asarray(x, dtype=np.uint8)]


def gemm_fp8(A, fmt_a: int, B, fmt_b: int, alpha: float = 1.0, beta: float = 0.0, C0=None,
             threads=None) -> np.ndarray:
    """fp64 alpha * dec(A) @ dec(B) + beta * C0."""
    return gemm(decode(A, fmt_a), decode(B, fmt_b), alpha, beta,
                None if C0 is None else to_f64(C0), threads)


def normwise_denominator_fp8(A, fmt_a, B, fmt_b, alpha=1.0, beta=0.0, C0=None, threads=None):
    """max(|alpha| sum_k |dec A||dec B| + |beta||C0|), the error scale."""
    from . import normwise_denominator
    return normwise_denominator(decode(A, fmt_a), decode(B, fmt_b), alpha, beta,
                                None if C0 is None else to_f64(C0), threads)
