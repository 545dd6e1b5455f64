"""Algorithmic work and traffic of one GEMM launch, and roofline arithmetic.

Used by the benchmark to turn a measured kernel duration into achieved
TFLOP/s or GB/s and a fraction of the roof.

* work: 2MNK FLOPs ("CUDA 算子工程 ch.10 朴素 GEMM 与 Roofline 分析", 10.3.1);
* algorithmic HBM bytes: A and B read once, C written once, and C read once
  more when beta != 0 (section 10.3.1 of that page; "Kernel 性能从何而来",
  section "GEMM", which drops the C read only for beta = 0);
* roof: min(P_compute, BW x AI) ("从模型计算到 GPU 执行", section 5.2).
"""
from __future__ import annotations


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * int(M) * int(N) * int(K)


def gemm_bytes(M: int, N: int, K: int, in_bytes: int, out_bytes: int,
               read_c: bool) -> int:
    """Bytes a GEMM must move: inputs of ``in_bytes``, C of ``out_bytes``."""
    M, N, K = int(M), int(N), int(K)
    inputs = in_bytes * (M * K + K * N)
    c_traffic = out_bytes * M * N * (2 if read_c else 1)
    return inputs + c_traffic


def gemm_ai(M: int, N: int, K: int, in_bytes: int, out_bytes: int,
            read_c: bool) -> float:
    return gemm_flops(M, N, K) / gemm_bytes(M, N, K, in_bytes, out_bytes, read_c)


def roof(p_compute: float, bandwidth: float, ai: float) -> float:
    return min(p_compute, bandwidth * ai)


def ridge(p_compute: float, bandwidth: float) -> float:
    return p_compute / bandwidth


def stage_tile_ai(bm: int, bn: int, bk: int, s: int) -> float:
    """A/B global-memory AI of one K-stage of a bm x bn CTA tile."""
    return (2.0 * bm * bn * bk) / (s * (bm * bk + bk * bn))


def fp32_peak(sms: int, clock_hz: float, lanes_per_sm: int = 128) -> float:
    """FP32 CUDA-core peak: every lane retires one FMA (2 FLOPs) per clock."""
    return sms * lanes_per_sm * 2.0 * clock_hz
