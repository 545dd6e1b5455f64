"""Closed-form work, traffic and roofline formulas of the pages -- TEST INFRASTRUCTURE ONLY.

Each function restates one formula, with the passage it follows.  The
benchmark computes its own algorithmic counts in the product package; the
tests pin both against the numbers the pages print.
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int) -> int:
    """2MNK: one multiply-add counts as two floating-point operations.

    "CUDA 算子工程 ch.10", section 10.3.1 (kernel-level count) and
    "Kernel 性能从何而来", section "Roofline 模型" (FMA = 2 FLOPs).
    """
    return 2 * M * N * K


def gemm_ideal_bytes(M: int, N: int, K: int, s: int, read_c: bool = False) -> int:
    """Ideal HBM traffic: A and B read once, C written once, elements of s bytes.

    "CUDA 算子工程 ch.10", section 10.3.1: s*(MK + KN + MN).  When beta != 0 the
    old C must also be read once (the count in "Kernel 性能从何而来", section
    "GEMM", leaves it out only because it assumes beta = 0).
    """
    return s * (M * K + K * N + M * N + (M * N if read_c else 0))


def gemm_ideal_ai(M: int, N: int, K: int, s: int, read_c: bool = False) -> float:
    """AI_kernel = 2MNK / (s(MK + KN + MN)), section 10.3.1 of ch.10."""
    return gemm_flops(M, N, K) / gemm_ideal_bytes(M, N, K, s, read_c)


def thread_ai_naive(K: int) -> float:
    """Per-thread AI of the naive kernel, 2K / (4K + 4K + 4): section 10.3.1."""
    return (2 * K) / (4 * K + 4 * K + 4)


def stage_tile_ai(BM: int, BN: int, BK: int, s: int) -> float:
    """Per-K-stage A/B global-memory AI of a BM x BN CTA tile.

    "Kernel 性能从何而来", section "优化 Memory-Bound Kernel" (blocking): the stage
    does 2*BM*BN*BK FLOPs and loads s*(BM*BK + BK*BN) bytes.
    """
    return (2 * BM * BN * BK) / (s * (BM * BK + BK * BN))


def roof(p_compute: float, bandwidth: float, ai: float) -> float:
    """P_max = min(P_compute, BW * AI): "从模型计算到 GPU 执行", section 5.2."""
    return min(p_compute, bandwidth * ai)


def ridge(p_compute: float, bandwidth: float) -> float:
    """AI_critical = P_compute / BW: "从模型计算到 GPU 执行", section 5.2."""
    return p_compute / bandwidth


def peak_from_units(sms: int, clock_hz: float, flops_per_sm_per_clock: float) -> float:
    """Peak = SMs x clock x FLOPs per SM per clock ("CUDA 算子工程 ch.10", 10.4.2)."""
    return sms * clock_hz * flops_per_sm_per_clock


def mma_tile_flops(m: int, n: int, k: int) -> int:
    """FLOPs of one m x n x k matrix-multiply instruction (2*m*n*k), section 10.4.2."""
    return 2 * m * n * k


def naive_reads(n: int) -> int:
    """Logical element reads of an n x n GEMM without reuse: n^2 outputs x 2n.

    "从模型计算到 GPU 执行", section 4.3 (16 for 2x2, 128 for 4x4).
    """
    return n * n * (2 * n)


def tiled_reads(n: int) -> int:
    """Logical element reads when every input is loaded once: 2 n^2 (same section)."""
    return 2 * n * n
