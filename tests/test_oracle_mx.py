"""Pins of the block-scaled (MX / NVFP4) oracle: the values the format
definitions fix, agreement with torch's E8M0 and FP4 types, worked examples
with hand-computed results (ragged last block, each scale format), the
reduction to the FP8 GEMM at unit scales, linearity over scale blocks, and
exact rational brute force on tiny inputs."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8, mx


def test_e8m0_values():
    assert mx.decode_e8m0(127) == 1.0
    assert mx.decode_e8m0(128) == 2.0 and mx.decode_e8m0(126) == 0.5
    assert mx.decode_e8m0(0) == 2.0 ** -127
    assert mx.decode_e8m0(254) == 2.0 ** 127
    assert math.isnan(mx.decode_e8m0(255))


def test_e8m0_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = mx.decode_scales(codes.numpy(), mx.E8M0)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])


def test_e2m1_values():
    # the eight magnitudes of the format, codes 0..7, and their negatives
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert [mx.decode_e2m1(c) for c in range(8)] == want
    assert [mx.decode_e2m1(c) for c in range(8, 16)] == [-w for w in want]
    assert math.copysign(1.0, mx.decode_e2m1(8)) == -1.0   # negative zero


def test_e2m1_matches_torch():
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("torch has no FP4 type")
    # every byte holds two codes, low nibble first
    packed = torch.arange(256, dtype=torch.uint8)
    try:
        ref = packed.view(torch.float4_e2m1fn_x2).to(torch.float32)
    except Exception as e:   # conversion not implemented in this build
        pytest.skip(f"torch cannot convert FP4: {e}")
    ref = ref.reshape(-1).to(torch.float64).numpy()
    ours = mx.decode_elements(packed.numpy().reshape(1, 256), mx.E2M1).reshape(-1)
    assert ref.shape == ours.shape
    assert np.array_equal(ref, ours)


def test_ue4m3_scale_values():
    assert mx.decode_ue4m3(0x38) == 1.0
    assert mx.decode_ue4m3(0x30) == 0.5
    assert mx.decode_ue4m3(0x7E) == 448.0
    assert mx.decode_ue4m3(0x01) == 2.0 ** -9
    assert math.isnan(mx.decode_ue4m3(0x7F))
    assert math.isnan(mx.decode_ue4m3(0xB8))      # a sign bit is not a scale


def test_fp4_packing_low_nibble_first():
    assert mx.pack_fp4([[1, 2]]).tolist() == [[0x21]]
    assert mx.unpack_fp4(np.array([[0x21, 0x7F]], dtype=np.uint8), 3).tolist() == [[1, 2, 15]]
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 16, size=(5, 9))
    assert np.array_equal(mx.unpack_fp4(mx.pack_fp4(codes), 9), codes)


def test_mxfp8_worked_example_with_a_ragged_block():
    # K = 40: one block of 32 and a ragged block of 8.  A = 1.0 (E4M3 0x38)
    # everywhere, with scales 2 and 0.5; B = 2.0 (0x40) with scale 1:
    # C = 32 * (2 * 1) * 2 + 8 * (0.5 * 1) * 2 = 128 + 8 = 136
    A = np.full((1, 40), 0x38, dtype=np.uint8)
    sA = np.array([[128, 126]], dtype=np.uint8)
    B = np.full((40, 1), 0x40, dtype=np.uint8)
    sB = np.array([[127], [127]], dtype=np.uint8)
    C = mx.gemm_block_scaled(A, sA, B, sB, mx.E4M3, mx.E4M3, mx.E8M0, mx.MXFP8_BLOCK, 40, 1)
    assert C.tolist() == [[136.0]]


def test_mxfp4_and_nvfp4_worked_examples():
    # MXFP4: A = 6.0 (code 7) x 32 at scale 2^-2 -> 1.5; B = 1.5 (code 3) at
    # scale 1: C = 32 * 1.5 * 1.5 = 72
    A = mx.pack_fp4(np.full((1, 32), 7))
    B = mx.pack_fp4(np.full((32, 1), 3))        # one column: packed along n
    C = mx.gemm_block_scaled(A, np.array([[125]], np.uint8), B, np.array([[127]], np.uint8),
                             mx.E2M1, mx.E2M1, mx.E8M0, mx.MXFP4_BLOCK, 32, 1)
    assert C.tolist() == [[72.0]]
    # NVFP4: blocks of 16, E4M3 scales: A = 1.0 (code 2) at 0.5 (0x30),
    # B = 3.0 (code 5) at 1.0 (0x38): C = 16 * 0.5 * 3 = 24; a second block
    # of A at scale 448 (0x7E) with code 1 (0.5) adds 16 * 224 * 3 = 10752
    A = mx.pack_fp4(np.concatenate([np.full((1, 16), 2), np.full((1, 16), 1)], axis=1))
    B = mx.pack_fp4(np.full((32, 1), 5))
    sA = np.array([[0x30, 0x7E]], np.uint8)
    sB = np.array([[0x38], [0x38]], np.uint8)
    C = mx.gemm_block_scaled(A, sA, B, sB, mx.E2M1, mx.E2M1, mx.UE4M3, mx.NVFP4_BLOCK, 32, 1)
    assert C.tolist() == [[24.0 + 10752.0]]


@pytest.mark.parametrize("fa,fb", [(mx.E4M3, mx.E4M3), (mx.E5M2, mx.E4M3), (mx.E4M3, mx.E5M2)])
def test_unit_scales_reduce_to_the_fp8_gemm(fa, fb):
    rng = np.random.default_rng(1)
    M, N, K = 9, 11, 70
    A = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    B = rng.integers(0, 256, size=(K, N), dtype=np.uint8)
    # keep finite codes only (E4M3 0x7F/0xFF, E5M2 exponent 31 are not numbers)
    A[np.isnan(fp8.decode(A, fa)) | np.isinf(fp8.decode(A, fa))] = 0x38
    B[np.isnan(fp8.decode(B, fb)) | np.isinf(fp8.decode(B, fb))] = 0x38
    sA = np.full((M, 3), 127, np.uint8)
    sB = np.full((3, N), 127, np.uint8)
    got = mx.gemm_block_scaled(A, sA, B, sB, fa, fb, mx.E8M0, 32, K, N, 1.5, 0.0)
    assert np.array_equal(got, fp8.gemm_fp8(A, fa, B, fb, 1.5))


def test_a_block_scale_scales_exactly_that_blocks_contribution():
    rng = np.random.default_rng(2)
    M, N, K = 4, 6, 96
    A = mx.pack_fp4(rng.integers(0, 16, size=(M, K)))
    B = mx.pack_fp4(rng.integers(0, 16, size=(K, N)))
    sA = rng.integers(120, 134, size=(M, 3)).astype(np.uint8)
    sB = rng.integers(120, 134, size=(3, N)).astype(np.uint8)
    base = mx.gemm_block_scaled(A, sA, B, sB, mx.E2M1, mx.E2M1, mx.E8M0, 32, K, N)
    sA2 = sA.copy()
    sA2[2, 1] += 1                                   # doubles block 1 of row 2
    moved = mx.gemm_block_scaled(A, sA2, B, sB, mx.E2M1, mx.E2M1, mx.E8M0, 32, K, N)
    # the change is exactly block 1's part of row 2, computed on its own
    dA = mx.dequant_a(A, sA, mx.E2M1, mx.E8M0, 32, K)
    dB = mx.dequant_b(B, sB, mx.E2M1, mx.E8M0, 32, N)
    part = dA[2, 32:64] @ dB[32:64, :]
    assert np.array_equal(moved[2] - base[2], part)
    others = [r for r in range(M) if r != 2]
    assert np.array_equal(moved[others], base[others])


@pytest.mark.parametrize("seed", [3, 4])
def test_brute_force_rationals(seed):
    # exact Fractions, element by element and block by block, written without
    # the oracle's repeat/GEMM assembly
    rng = np.random.default_rng(seed)
    M, N, K, V = 3, 4, 37, 16
    a_codes = rng.integers(0, 16, size=(M, K))
    b_codes = rng.integers(0, 16, size=(K, N))
    sA = rng.integers(0x20, 0x48, size=(M, -(-K // V))).astype(np.uint8)
    sB = rng.integers(0x20, 0x48, size=(-(-K // V), N)).astype(np.uint8)
    got = mx.gemm_block_scaled(mx.pack_fp4(a_codes), sA, mx.pack_fp4(b_codes), sB,
                               mx.E2M1, mx.E2M1, mx.UE4M3, V, K, N)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = Fraction(mx.decode_e2m1(int(a_codes[m, k]))) * Fraction(mx.decode_ue4m3(int(sA[m, k // V])))
                b = Fraction(mx.decode_e2m1(int(b_codes[k, n]))) * Fraction(mx.decode_ue4m3(int(sB[k // V, n])))
                acc += a * b
            assert got[m, n] == float(acc)


def test_error_scale_bounds_the_result():
    rng = np.random.default_rng(5)
    M, N, K = 5, 7, 64
    A = rng.integers(0, 120, size=(M, K), dtype=np.uint8)   # finite positive E4M3
    B = rng.integers(0, 120, size=(K, N), dtype=np.uint8)
    sA = np.full((M, 2), 127, np.uint8)
    sB = np.full((2, N), 128, np.uint8)
    C = mx.gemm_block_scaled(A, sA, B, sB, mx.E4M3, mx.E4M3, mx.E8M0, 32, K, N)
    d = mx.normwise_denominator_block_scaled(A, sA, B, sB, mx.E4M3, mx.E4M3, mx.E8M0, 32, K, N)
    assert np.max(np.abs(C)) <= d
    assert d == np.max(C)   # all products are non-negative here
