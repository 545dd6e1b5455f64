"""Pins of the FP8 decoding: values the format definitions fix, the order of
the codes, and agreement with torch's float8 types on every byte."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_e4m3_special_values():
    d = lambda b: fp8.decode_byte(b, fp8.E4M3)
    assert d(0x00) == 0.0 and math.copysign(1, d(0x80)) == -1
    assert d(0x38) == 1.0                 # exponent 7 = bias, mantissa 0
    assert d(0x7E) == 448.0               # largest finite: 1.75 * 2^8
    assert d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6           # smallest normal
    assert d(0x07) == 7 / 8 * 2.0 ** -6   # largest subnormal
    assert d(0x01) == 2.0 ** -9           # smallest subnormal
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x3C) == 1.5 and d(0x40) == 2.0 and d(0xC4) == -3.0


def test_e5m2_special_values():
    d = lambda b: fp8.decode_byte(b, fp8.E5M2)
    assert d(0x3C) == 1.0
    assert d(0x7B) == 57344.0             # largest finite: 1.75 * 2^15
    assert d(0x7C) == math.inf and d(0xFC) == -math.inf
    assert all(math.isnan(d(b)) for b in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    assert d(0x04) == 2.0 ** -14          # smallest normal
    assert d(0x01) == 2.0 ** -16          # smallest subnormal
    assert d(0x3E) == 1.5 and d(0xC0) == -2.0


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_codes_are_ordered_and_symmetric(fmt):
    t = fp8.table(fmt)
    pos = t[:128][np.isfinite(t[:128])]
    assert np.all(np.diff(pos) > 0)                    # codes 0..127 increase
    finite = np.isfinite(t[:128])
    assert np.array_equal(t[128:][finite], -t[:128][finite])   # sign bit only flips


@pytest.mark.parametrize("fmt,dtype", [(fp8.E4M3, "float8_e4m3fn"), (fp8.E5M2, "float8_e5m2")])
def test_every_code_matches_torch(fmt, dtype):
    if not hasattr(torch, dtype):
        pytest.skip(f"torch has no {dtype}")
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(getattr(torch, dtype)).to(torch.float64).numpy()
    got = fp8.decode(codes, fmt)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp8_gemm_is_the_gemm_of_the_decoded_values():
    # small integers are exact in both formats: the FP8 GEMM of their codes
    # equals the integer GEMM
    rng = np.random.default_rng(5)
    Ai = rng.integers(-8, 9, size=(5, 7)).astype(np.float64)
    Bi = rng.integers(-8, 9, size=(7, 4)).astype(np.float64)
    enc = {v: b for b in range(256) for v in [fp8.decode_byte(b, fp8.E4M3)]
           if not math.isnan(v) and not (v == 0 and b & 0x80)}
    A = np.vectorize(lambda v: enc[v])(Ai).astype(np.uint8)
    enc5 = {v: b for b in range(256) for v in [fp8.decode_byte(b, fp8.E5M2)]
            if not math.isnan(v) and not math.isinf(v) and not (v == 0 and b & 0x80)}
    B = np.vectorize(lambda v: enc5[v])(Bi).astype(np.uint8)
    got = fp8.gemm_fp8(A, fp8.E4M3, B, fp8.E5M2, 0.5, 0.0)
    assert np.array_equal(got, 0.5 * (Ai @ Bi))
