"""Pins of the closed-form FLOP / traffic / roofline formulas to the pages' numbers.

Both restatements are checked: the oracle's (``oracle.roofline_ref``) and the
one the benchmark uses (``roofline_driven_optimisation_gb300.roofline``).
"""
import os

import pytest

from conftest import GOLDEN
from oracle import roofline_ref as R
from roofline_driven_optimisation_gb300 import roofline as P


def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "roofline_numbers.txt"), encoding="utf-8") as f:
        for ln in f:
            if not ln.strip() or ln.startswith("#"):
                continue
            key, val, tol, _src = [x.strip() for x in ln.split("|")]
            vals[key] = (float(val), float(tol))
    return vals


G = _golden()


def _check(key, value):
    want, tol = G[key]
    if tol == 0:
        assert value == want, (key, value, want)
    else:
        assert abs(value - want) <= tol * abs(want), (key, value, want)


def test_ai_kernel_fp32_4096():
    _check("ai_kernel_fp32_4096", R.gemm_ideal_ai(4096, 4096, 4096, 4))
    _check("ai_kernel_fp32_4096", P.gemm_ai(4096, 4096, 4096, 4, 4, read_c=False))


def test_ai_thread_limit():
    _check("ai_thread_naive_limit", R.thread_ai_naive(10 ** 7))


def test_ridges():
    _check("ridge_h100_fp32", R.ridge(67e12, 3.35e12))
    _check("ridge_h100_bf16", R.ridge(989e12, 3.35e12))
    _check("hypo_ridge", R.ridge(20e12, 500e9))
    _check("b200_ridge", R.ridge(2e15, 8e12))
    _check("ridge_h100_bf16", P.ridge(989e12, 3.35e12))


def test_hypothetical_roofline():
    _check("hypo_roof_ai1_tflops", R.roof(20e12, 500e9, 1.0) / 1e12)
    _check("hypo_roof_ai10_tflops", R.roof(20e12, 500e9, 10.0) / 1e12)
    _check("hypo_roof_ai10_tflops", P.roof(20e12, 500e9, 10.0) / 1e12)
    # right of the ridge the compute roof holds
    assert R.roof(20e12, 500e9, 1000.0) == 20e12


def test_stage_tile_ai():
    _check("stage_flops_16x16", 2 * 16 * 16 * 64)
    _check("stage_bytes_16x16", 2 * (16 * 64 + 64 * 16))
    _check("stage_ai_16x16", R.stage_tile_ai(16, 16, 64, 2))
    _check("stage_flops_64x64", 2 * 64 * 64 * 64)
    _check("stage_bytes_64x64", 2 * (64 * 64 + 64 * 64))
    _check("stage_ai_64x64", R.stage_tile_ai(64, 64, 64, 2))
    # B_M = B_N = B reduces to B / s
    assert R.stage_tile_ai(128, 128, 64, 2) == 128 / 2
    assert P.stage_tile_ai(64, 64, 64, 2) == 32


def test_tensor_core_peak_derivation():
    _check("mma_m16n8k16_flops", R.mma_tile_flops(16, 8, 16))
    per_sm_per_clock = 4 * R.mma_tile_flops(16, 8, 16) / 4   # 4 TCs, ~4 cycles each
    _check("h100_bf16_peak_tflops", R.peak_from_units(132, 1.83e9, per_sm_per_clock) / 1e12)


def test_logical_read_counts():
    _check("naive_reads_2x2", R.naive_reads(2))
    _check("tiled_reads_2x2", R.tiled_reads(2))
    _check("naive_reads_4x4", R.naive_reads(4))
    _check("tiled_reads_4x4", R.tiled_reads(4))


def test_reuse_factors():
    _check("reuse_block_128x128", (128 * 128) / (128 + 128))
    _check("reuse_warp_64x32", (64 * 32) / (64 + 32))
    _check("thread_tile_4x4_ai", (2 * 4 * 4) / (4 * (4 + 4)))


def test_flops_and_bytes():
    assert R.gemm_flops(4096, 4096, 4096) == 2 * 4096 ** 3
    assert P.gemm_flops(4096, 4096, 4096) == 2 * 4096 ** 3
    # beta != 0 adds one read of C; bf16 in, fp32 out
    assert R.gemm_ideal_bytes(2, 3, 4, 4, read_c=True) == 4 * (8 + 12 + 6 + 6)
    assert P.gemm_bytes(2, 3, 4, 2, 4, read_c=True) == 2 * (8 + 12) + 4 * (6 + 6)
    # square bf16 GEMM at 4096: N/3 = 1365.3 ("~1300" in the AI table of ch.4, 4.6)
    assert abs(R.gemm_ideal_ai(4096, 4096, 4096, 2) - 4096 / 3) < 1e-9


def test_gb300_unit_counts():
    # FP32 CUDA-core peak: SMs x 128 lanes x 2 FLOPs x clock
    assert P.fp32_peak(152, 2070e6) == pytest.approx(152 * 128 * 2 * 2.07e9)
