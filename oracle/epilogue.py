"""Elementwise epilogues in fp64 -- TEST INFRASTRUCTURE ONLY.

The fused-epilogue GEMM is  C = act(alpha*A*B + beta*C0 + bias)  with bias[n]
added to every row ("Kernel 性能从何而来", section "优化 Memory-Bound Kernel":
GEMM fused with an elementwise epilogue).  The activations are their plain
definitions:

    relu(z) = max(z, 0)
    silu(z) = z * sigmoid(z) = z / (1 + exp(-z))
    gelu(z) = z * Phi(z) = 0.5 z (1 + erf(z / sqrt(2)))       (exact, erf form)
    swiglu(g, u) = silu(g) * u                                  (LLaMA FFN gate/up)
"""
from __future__ import annotations

import math

import numpy as np

from . import gemm, to_f64

NONE, RELU, SILU, GELU = 0, 1, 2, 3


def _erf(x: np.ndarray) -> np.ndarray:
    try:
        from scipy.special import erf
        return erf(x)
    except ImportError:  # pragma: no cover - scipy is present on both machines
        return np.vectorize(math.erf, otypes=[np.float64])(x)


def activate(z, act: int) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    if act == NONE:
        return z.copy()
    if act == RELU:
        return np.maximum(z, 0.0)
    if act == SILU:
        with np.errstate(over="ignore"):
            return z / (1.0 + np.exp(-z))
    if act == GELU:
        return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))
    raise ValueError(act)


def gemm_epilogue(A, B, alpha=1.0, beta=0.0, C0=None, bias=None, act=NONE, threads=None):
    """fp64 act(alpha*A@B + beta*C0 + bias)."""
    z = gemm(A, B, alpha, beta, C0, threads)
    if bias is not None:
        z = z + to_f64(bias).reshape(1, -1)
    return activate(z, act)


def swiglu(A, Bgate, Bup, threads=None):
    """fp64 silu(A@Bgate) * (A@Bup)."""
    g = gemm(A, Bgate, 1.0, 0.0, None, threads)
    u = gemm(A, Bup, 1.0, 0.0, None, threads)
    return activate(g, SILU) * u


# max over z of d/dz silu(z) = sigmoid(z) (1 + z (1 - sigmoid(z))), about
# 1.0998 near z = 2.40; 1.1 bounds it
SILU_SLOPE_BOUND = 1.1


def swiglu_error_scale(A, Bgate, Bup, threads=None) -> float:
    """Scale for the normwise error of a computed swiglu(A, Bgate, Bup).

    With g = A@Bgate and u = A@Bup each accumulated with an error of at most
    e * sum_k |A||B| (rounding of the products and sums), the first-order
    error of silu(g) * u is at most
        e * (SILU_SLOPE_BOUND |u| sum_k|A||Bgate| + |silu(g)| sum_k|A||Bup|),
    and the final rounding of silu(g) * u is bounded by the same scale (since
    |u| <= sum_k |A||Bup|).  Returns the max over elements of the bracket.
    """
    g = gemm(A, Bgate, 1.0, 0.0, None, threads)
    u = gemm(A, Bup, 1.0, 0.0, None, threads)
    Aa = np.abs(to_f64(A))
    Sg = gemm(Aa, np.abs(to_f64(Bgate)), 1.0, 0.0, None, threads)
    Su = gemm(Aa, np.abs(to_f64(Bup)), 1.0, 0.0, None, threads)
    S = SILU_SLOPE_BOUND * np.abs(u) * Sg + np.abs(activate(g, SILU)) * Su
    return float(S.max()) if S.size else 0.0
