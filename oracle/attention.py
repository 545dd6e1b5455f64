"""Attention in fp64 -- TEST INFRASTRUCTURE ONLY.

"从模型计算到 GPU 执行：读懂算子、Kernel 与 GPU 性能", section 1.2: attention is
softmax(Q K^T / sqrt(d)) V, computed in the steps

    S = Q K^T,   S = S * scale (scale = 1/sqrt(d)),   P = softmax(S) row by row,   O = P V.

Shapes follow the usual multi-head layout: Q is [B][Hq][Sq][d], K and V are
[B][Hkv][Sk][d] with Hq a multiple of Hkv (query head h reads key/value head
h // (Hq / Hkv); Hkv = Hq is plain multi-head attention), O is [B][Hq][Sq][d].
With `causal`, query i sees key j only when j <= i + (Sk - Sq) (the last
query row is aligned with the last key); masked scores are -inf before the
softmax.  A row with no visible key gives O = 0.
"""
from __future__ import annotations

import math

import numpy as np

from . import to_f64


def _mask(Sq: int, Sk: int, causal: bool) -> np.ndarray:
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    return (j <= i + (Sk - Sq)) if causal else np.ones((Sq, Sk), dtype=bool)


def _softmax_rows(S: np.ndarray, visible: np.ndarray) -> np.ndarray:
    S = np.where(visible, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    E = np.where(visible, np.exp(S - m), 0.0)
    den = E.sum(axis=1, keepdims=True)
    return np.divide(E, den, out=np.zeros_like(E), where=den > 0)


def attention(Q, K, V, scale: float | None = None, causal: bool = False) -> np.ndarray:
    """fp64 O = softmax(Q K^T * scale) V for [B][H][S][d] arrays."""
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    B, Hq, Sq, d = Q.shape
    Hkv, Sk = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    vis = _mask(Sq, Sk, causal)
    O = np.zeros((B, Hq, Sq, V.shape[3]))
    for b in range(B):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            S = Q[b, h] @ K[b, kv].T
            S = S * scale
            P = _softmax_rows(S, vis)
            O[b, h] = P @ V[b, kv]
    return O


def error_scale(Q, K, V, scale: float | None = None, causal: bool = False) -> float:
    """max over (b, h, i, c) of sum_j P[i][j] |V[j][c]|: the size of each output
    element's weighted average, the scale its error is measured against."""
    Q, K, V = to_f64(Q), to_f64(K), to_f64(V)
    B, Hq, Sq, d = Q.shape
    Hkv, Sk = K.shape[1], K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    vis = _mask(Sq, Sk, causal)
    worst = 0.0
    for b in range(B):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            P = _softmax_rows((Q[b, h] @ K[b, kv].T) * scale, vis)
            worst = max(worst, float((P @ np.abs(V[b, kv])).max(initial=0.0)))
    return worst
