"""INT4 weights in fp64 -- TEST INFRASTRUCTURE ONLY.

"CUDA 算子工程 ch.4 内存层级与代价表", section 4.5.3: an INT4 matrix holds two
4-bit codes per byte, the first element in the low nibble and the second in
the high nibble, and dequantisation multiplies each code by a scale.  Written
out for a K x N weight with codes q (0..15):

    W[k][n] = s[k // G][n] * (q[k][n] - z)

with one scale per group of G consecutive rows and per column (bf16; the
pages' single scale is the case of equal scales), and one integer zero point
z (the pages' code is z = 0).  W is exact in fp32 (a bf16 scale times an
integer of at most 4 bits); the dequantised weight the GEMM consumes is that
value rounded once to bf16 (round to nearest even), the type of the MMA's
other operand.  Byte j of row k packs columns 2j (bits 0-3) and 2j+1 (bits
4-7).
"""
from __future__ import annotations

import numpy as np
import torch

from . import gemm, to_f64


def unpack(q_bytes, N: int) -> np.ndarray:
    """K x N codes (int64) from K x ceil(N/2) packed bytes."""
    b = np.asarray(q_bytes.cpu().numpy() if hasattr(q_bytes, "cpu") else q_bytes, dtype=np.uint8)
    codes = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.int64)
    codes[:, 0::2] = b & 0x0F
    codes[:, 1::2] = b >> 4
    return codes[:, :N]


def dequant_exact(q_bytes, scales, N: int, group: int, zero: int) -> np.ndarray:
    """fp64 s[k // G][n] * (q[k][n] - z) (exact)."""
    codes = unpack(q_bytes, N)
    s = to_f64(scales)[:, :N]
    rows = np.arange(codes.shape[0]) // group
    return s[rows, :] * (codes - zero).astype(np.float64)


def dequant_bf16(q_bytes, scales, N: int, group: int, zero: int) -> torch.Tensor:
    """The dequantised weight as bf16: the exact value rounded once (RNE)."""
    w = torch.from_numpy(dequant_exact(q_bytes, scales, N, group, zero))
    # the exact value has at most 12 significant bits, so fp64 -> fp32 is
    # exact and the single rounding happens in fp32 -> bf16
    return w.to(torch.float32).to(torch.bfloat16)


def gemm_w4(A, q_bytes, scales, N: int, group: int, zero: int, alpha=1.0, beta=0.0, C0=None,
            threads=None) -> np.ndarray:
    """fp64 alpha * A @ W + beta * C0 with W the bf16 dequantised weight."""
    W = dequant_bf16(q_bytes, scales, N, group, zero)
    return gemm(A, W, alpha, beta, None if C0 is None else to_f64(C0), threads)
