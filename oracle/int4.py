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


def gemm_w4_exact(A, q_bytes, scales, N: int, group: int, zero: int, alpha=1.0, beta=0.0, C0=None,
                  threads=None) -> np.ndarray:
    """fp64 alpha * A @ W + beta * C0 with W = s * (q - z) exact (the INT4 GEMM
    that never rounds the weight: the integers q - z enter the products and
    each group's sum is scaled)."""
    W = dequant_exact(q_bytes, scales, N, group, zero)
    return gemm(A, W, alpha, beta, None if C0 is None else to_f64(C0), threads)


# Order of the eight codes of one 32-bit word in the K-packed layout: slot s
# (bits 4s..4s+3) holds the code of k = 8j + SLOT_K[s], so that bits 0-3 and
# 16-19 of (word >> 4i) are the codes of k = 8j + 2i and 8j + 2i + 1.
SLOT_K = (0, 2, 4, 6, 1, 3, 5, 7)


def repack_kmajor(q_bytes, K: int, N: int) -> np.ndarray:
    """K-packed layout of a K x N weight: row n holds ceil(K/8) little-endian
    32-bit words, word j packing the codes of k = 8j..8j+7 in the slot order
    SLOT_K (codes past K are 0).  Returns N x 4*ceil(K/8) bytes."""
    codes = unpack(q_bytes, N)                   # K x N
    words = (K + 7) // 8
    padded = np.zeros((words * 8, N), dtype=np.int64)
    padded[:K] = codes
    out = np.zeros((N, words), dtype=np.uint64)
    for s, dk in enumerate(SLOT_K):
        out |= (padded[dk::8].T.astype(np.uint64) << np.uint64(4 * s))
    return out.astype("<u4").view(np.uint8).reshape(N, 4 * words)


# Tiled K-packed layout: W is cut into tiles of TILE_N columns by TILE_K rows
# of K, stored one after another (column tiles outer, K tiles inner), each
# tile TILE_N x TILE_K/2 bytes with column n's codes for its TILE_K rows of K
# as TILE_K/8 words in the SLOT_K order.  Tiles past N or K are zero-filled.
TILE_N, TILE_K = 128, 64


def tiled_bytes(K: int, N: int) -> int:
    return -(-N // TILE_N) * -(-K // TILE_K) * TILE_N * TILE_K // 2


def repack_tiled(q_bytes, K: int, N: int) -> np.ndarray:
    """The tiled K-packed layout as a flat uint8 array of tiled_bytes(K, N)."""
    tn, tk = -(-N // TILE_N), -(-K // TILE_K)
    rows = repack_kmajor(q_bytes, K, N)                         # N x 4*ceil(K/8)
    full = np.zeros((tn * TILE_N, tk * TILE_K // 2), dtype=np.uint8)
    full[:N, : rows.shape[1]] = rows
    tiles = full.reshape(tn, TILE_N, tk, TILE_K // 2).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(tiles).reshape(-1)