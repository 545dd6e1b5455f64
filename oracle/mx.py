"""Block-scaled low-precision inputs in fp64 -- TEST INFRASTRUCTURE ONLY.

"Kernel 性能从何而来", section "优化 Memory-Bound Kernel": narrower data types
(fp8, fp4) cut the bytes moved per FLOP, and the block-scaled fp8/fp4 formats
carry scale factors alongside the elements.  The plain reading of a
block-scaled GEMM is the GEMM of the values the blocks encode:

    C = alpha * dec(A) * dec(B) + beta * C0,
    dec(A)[m, k] = scale_A[m, k / V] * elem(A[m, k])
    dec(B)[k, n] = scale_B[k / V, n] * elem(B[k, n])

where the scale blocks run along K, the reduction dimension, V elements
each.  The formats are those of the OCP Microscaling (MX) specification and
NVIDIA's NVFP4:

  MXFP8  elements E4M3 or E5M2 (as in oracle.fp8), V = 32, scale E8M0;
  MXFP4  elements E2M1, V = 32, scale E8M0;
  NVFP4  elements E2M1, V = 16, scale an unsigned E4M3 byte (sign bit 0),
         times one fp32 tensor scale that the caller folds into alpha.

  E8M0: eight exponent bits, bias 127, no sign and no mantissa: code e is
        2^(e - 127) for e = 0..254; e = 255 is NaN.
  E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
        subnormal (m/2 * 2^0); no infinities or NaN; the magnitudes are
        0, 0.5, 1, 1.5, 2, 3, 4, 6.

Every decoded value (a power of two times an FP8 or FP4 value, or an FP8
value times an FP8 value for NVFP4) is exact in fp64, so the oracle GEMM of
dec(A), dec(B) is exact up to its own fp64 rounding.

Layout of the codes (the plain reading; the pages give none): FP8 elements
one per byte, row-major; FP4 elements two per byte along the contiguous
dimension, the first element in the low nibble (as the INT4 codes of
oracle.int4 and the pages' dequantisation example).  A's scales are an
M x ceil(K/V) byte matrix, B's a ceil(K/V) x N byte matrix.  A ragged last
block covers the K % V remaining elements with its own scale.
"""
from __future__ import annotations

import math

import numpy as np

from . import fp8, gemm, normwise_denominator, to_f64

# element formats
E4M3, E5M2, E2M1 = fp8.E4M3, fp8.E5M2, 2
# scale formats
E8M0, UE4M3 = 0, 1

MXFP8_BLOCK = 32
MXFP4_BLOCK = 32
NVFP4_BLOCK = 16


def decode_e8m0(code: int) -> float:
    """Value of one E8M0 scale byte: 2^(code - 127); 255 is NaN."""
    if code == 255:
        return math.nan
    return math.ldexp(1.0, code - 127)


def decode_e2m1(code: int) -> float:
    """Value of one E2M1 nibble from the field definitions."""
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return sign * (m / 2.0)            # subnormal: 0.m * 2^(1 - bias), bias 1
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


def decode_ue4m3(code: int) -> float:
    """Value of one unsigned E4M3 scale byte (NVFP4): the E4M3 value of the
    byte with its sign bit clear; a set sign bit is not a valid scale (NaN)."""
    if code & 0x80:
        return math.nan
    return fp8.decode_byte(code, fp8.E4M3)


_E8M0 = np.array([decode_e8m0(c) for c in range(256)], dtype=np.float64)
_UE4M3 = np.array([decode_ue4m3(c) for c in range(256)], dtype=np.float64)
_E2M1 = np.array([decode_e2m1(c) for c in range(16)], dtype=np.float64)


def _np_u8(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.uint8)


def decode_scales(s, scale_fmt: int) -> np.ndarray:
    """fp64 values of an array of scale bytes."""
    t = _E8M0 if scale_fmt == E8M0 else _UE4M3
    return t[_np_u8(s)]


def unpack_fp4(packed, cols: int) -> np.ndarray:
    """FP4 codes (0..15) of a row-major array of packed bytes, two codes per
    byte along the last dimension (low nibble first), cut to `cols`."""
    p = _np_u8(packed)
    lo, hi = p & 0xF, p >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    return codes[..., :cols]


def pack_fp4(codes) -> np.ndarray:
    """Inverse of unpack_fp4: codes (0..15) two per byte, low nibble first
    (an odd last column is padded with code 0)."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    if c.shape[-1] % 2:
        c = np.concatenate([c, np.zeros((*c.shape[:-1], 1), dtype=np.uint8)], axis=-1)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def decode_elements(x, elem_fmt: int, cols: int | None = None) -> np.ndarray:
    """fp64 values of the elements: FP8 bytes, or packed FP4 (then `cols`
    gives the unpacked length of the last dimension)."""
    if elem_fmt == E2M1:
        p = _np_u8(x)
        return _E2M1[unpack_fp4(p, cols if cols is not None else 2 * p.shape[-1])]
    return fp8.decode(x, elem_fmt)


def dequant_a(codes, scales, elem_fmt: int, scale_fmt: int, block: int, K: int) -> np.ndarray:
    """dec(A) for A (M x K): element m, k times scale[m, k // block]."""
    v = decode_elements(codes, elem_fmt, K)[:, :K]
    s = decode_scales(scales, scale_fmt)
    nb = -(-K // block)
    if s.shape[1] < nb:
        raise ValueError("A needs ceil(K / block) scales per row")
    return v * np.repeat(s[:, :nb], block, axis=1)[:, :K]


def dequant_b(codes, scales, elem_fmt: int, scale_fmt: int, block: int, N: int) -> np.ndarray:
    """dec(B) for B (K x N): element k, n times scale[k // block, n]."""
    v = decode_elements(codes, elem_fmt, N)[:, :N]
    K = v.shape[0]
    s = decode_scales(scales, scale_fmt)
    nb = -(-K // block)
    if s.shape[0] < nb:
        raise ValueError("B needs ceil(K / block) rows of scales")
    return v * np.repeat(s[:nb, :N], block, axis=0)[:K, :]


def gemm_block_scaled(A, sA, B, sB, elem_a: int, elem_b: int, scale_fmt: int, block: int,
                      K: int, N: int, alpha: float = 1.0, beta: float = 0.0, C0=None,
                      threads=None) -> np.ndarray:
    """fp64 alpha * dec(A) @ dec(B) + beta * C0 (the oracle GEMM of the
    decoded values)."""
    dA = dequant_a(A, sA, elem_a, scale_fmt, block, K)
    dB = dequant_b(B, sB, elem_b, scale_fmt, block, N)
    return gemm(dA, dB, alpha, beta, None if C0 is None else to_f64(C0), threads)


def normwise_denominator_block_scaled(A, sA, B, sB, elem_a, elem_b, scale_fmt, block, K, N,
                                      alpha=1.0, beta=0.0, C0=None, threads=None) -> float:
    """max(|alpha| sum_k |dec A||dec B| + |beta||C0|), the error scale."""
    dA = dequant_a(A, sA, elem_a, scale_fmt, block, K)
    dB = dequant_b(B, sB, elem_b, scale_fmt, block, N)
    return normwise_denominator(dA, dB, alpha, beta, None if C0 is None else to_f64(C0), threads)
