"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and rounds them to the element type the
GPU receives.  It holds none of the GEMM arithmetic, so both the CUDA path and
the CPU oracle can take their operands from it.

Workloads (the shapes and distributions the pages analyse):

* ``fp32_256``   FP32 SGEMM, M=N=K=256, alpha=1, beta=0, A,B ~ U[-1,1), seed 0.
* ``fp32_4096``  FP32 SGEMM, M=N=K=4096, alpha=1.5, beta=0.5, A,B,C0 ~ U[-1,1),
  seed 1 -- the 683 FLOP/byte case of "CUDA 算子工程 ch.10, 朴素 GEMM 与
  Roofline 分析" section 10.3.1.
* ``bf16_4096`` / ``bf16_8192``  BF16 GEMM with fp32 accumulation, alpha=1,
  beta=0, A,B ~ normal(0, 1/sqrt(K)) rounded to bf16, seed 2.
* ``prefill_<w>``  LLaMA-7B-shaped weight GEMMs at M=2048 tokens (d=4096,
  FFN 11008, vocab 32000 as in section 10.1 of the same page): X ~ N(0,1),
  W ~ N(0, 0.02), rounded to bf16, seed 3, alpha=1, beta=0.
* ``decode_m<M>_<w>``  the same weight shapes with M in {1, 4, 16} tokens,
  W ~ N(0, 0.02), X ~ N(0, 1), C0 ~ N(0, 1), seed 4, beta=1 (residual add).

Every case draws from its own ``torch.Generator`` seeded with the case's seed,
in the order A, B, C0, in fp32 on the CPU; bf16 cases are then rounded with
round-to-nearest-even (``Tensor.to(torch.bfloat16)``).  "normal(0, s)" means
standard deviation s.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# LLaMA-7B weight shapes (K, N) for the per-layer GEMMs and the LM head.
LLAMA7B_WEIGHTS = {
    "qkv": (4096, 12288),
    "o": (4096, 4096),
    "gate": (4096, 11008),
    "up": (4096, 11008),
    "down": (11008, 4096),
    "lm": (4096, 32000),
}
DECODE_M = (1, 4, 16)
PREFILL_M = 2048


@dataclasses.dataclass(frozen=True)
class CaseSpec:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    in_dtype: str          # "f32" or "bf16"
    seed: int
    dist: str              # "uniform", "normal_invsqrtk", "llama"
    c0: bool               # whether an initial C is drawn


@dataclasses.dataclass
class Case:
    spec: CaseSpec
    A: torch.Tensor        # M x K, row-major, CPU, element type the GPU gets
    B: torch.Tensor        # K x N
    C0: Optional[torch.Tensor]  # M x N or None (beta == 0)


def _specs() -> dict:
    s = {}
    s["fp32_256"] = CaseSpec("fp32_256", 256, 256, 256, 1.0, 0.0, "f32", 0, "uniform", False)
    s["fp32_4096"] = CaseSpec("fp32_4096", 4096, 4096, 4096, 1.5, 0.5, "f32", 1, "uniform", True)
    for n in (4096, 8192):
        s[f"bf16_{n}"] = CaseSpec(f"bf16_{n}", n, n, n, 1.0, 0.0, "bf16", 2, "normal_invsqrtk", False)
    for w, (K, N) in LLAMA7B_WEIGHTS.items():
        s[f"prefill_{w}"] = CaseSpec(f"prefill_{w}", PREFILL_M, N, K, 1.0, 0.0, "bf16", 3, "llama", False)
        for m in DECODE_M:
            s[f"decode_m{m}_{w}"] = CaseSpec(f"decode_m{m}_{w}", m, N, K, 1.0, 1.0, "bf16", 4, "llama", True)
    return s


SPECS = _specs()


def spec(name: str) -> CaseSpec:
    return SPECS[name]


def _draw(spec_: CaseSpec, gen: torch.Generator, which: str, rows: int, cols: int) -> torch.Tensor:
    shape = (rows, cols)
    if spec_.dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if spec_.dist == "normal_invsqrtk":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * (1.0 / math.sqrt(spec_.K))
    if spec_.dist == "llama":
        # activations and the initial C are N(0,1); weights N(0, 0.02)
        std = 0.02 if which == "B" else 1.0
        return torch.randn(shape, generator=gen, dtype=torch.float32) * std
    raise ValueError(spec_.dist)


def round_to(x: torch.Tensor, in_dtype: str) -> torch.Tensor:
    """Round fp32 values to the GPU element type (RNE for bf16)."""
    if in_dtype == "f32":
        return x.contiguous()
    if in_dtype == "bf16":
        return x.to(torch.bfloat16).contiguous()
    raise ValueError(in_dtype)


def make(spec_or_name, M: Optional[int] = None, N: Optional[int] = None,
         K: Optional[int] = None) -> Case:
    """Draw the operands of a workload (optionally at a reduced M/N/K).

    The overrides keep the seed and distributions of the named workload, which
    is how parity tests at small sizes mirror the full-size configuration.
    """
    sp = SPECS[spec_or_name] if isinstance(spec_or_name, str) else spec_or_name
    if M is not None or N is not None or K is not None:
        sp = dataclasses.replace(sp, M=sp.M if M is None else M,
                                 N=sp.N if N is None else N,
                                 K=sp.K if K is None else K)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(sp.seed)
    A = round_to(_draw(sp, gen, "A", sp.M, sp.K), sp.in_dtype)
    B = round_to(_draw(sp, gen, "B", sp.K, sp.N), sp.in_dtype)
    C0 = None
    if sp.c0:
        C0 = _draw(sp, gen, "C", sp.M, sp.N)
        # the initial C has the element type of the output it is added into
        C0 = round_to(C0, sp.in_dtype)
    return Case(sp, A, B, C0)


def random_matrix(rows: int, cols: int, seed: int, dtype: str = "f32",
                  dist: str = "uniform", std: float = 1.0) -> torch.Tensor:
    """A seeded matrix for edge-case tests (odd shapes, padding, scaling)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if dist == "uniform":
        x = torch.rand((rows, cols), generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn((rows, cols), generator=gen, dtype=torch.float32) * std
    elif dist == "int":
        x = torch.randint(-8, 9, (rows, cols), generator=gen).to(torch.float32)
    else:
        raise ValueError(dist)
    return round_to(x, dtype)


def device_uniform(rows: int, cols: int, seed: int, device, dtype: str = "bf16",
                   block_rows: int = 4096) -> torch.Tensor:
    """A seeded U[-1, 1) matrix drawn on `device` itself, a block of rows at a
    time, for operands too large to draw on the host and copy over; the same
    seed on the same kind of device gives the same values."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    out = torch.empty((rows, cols), dtype=tdt, device=device)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        x = torch.rand((r1 - r0, cols), generator=gen, device=device, dtype=torch.float32)
        out[r0:r1] = (x * 2.0 - 1.0).to(tdt)
    return out


@dataclasses.dataclass
class SwigluCase:
    A: torch.Tensor        # M x K activations, bf16, CPU
    Bgate: torch.Tensor    # K x N gate projection, bf16
    Bup: torch.Tensor      # K x N up projection, bf16


def make_swiglu(M: int, N: int = LLAMA7B_WEIGHTS["gate"][1], K: int = LLAMA7B_WEIGHTS["gate"][0],
                seed: int = 5) -> SwigluCase:
    """Operands of the fused FFN gate/up pair: activations N(0,1), both
    weights N(0, 0.02) (the LLaMA recipe of the other workloads), bf16."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    A = round_to(torch.randn((M, K), generator=gen, dtype=torch.float32), "bf16")
    Bg = round_to(torch.randn((K, N), generator=gen, dtype=torch.float32) * 0.02, "bf16")
    Bu = round_to(torch.randn((K, N), generator=gen, dtype=torch.float32) * 0.02, "bf16")
    return SwigluCase(A, Bg, Bu)


FP8_E4M3, FP8_E5M2 = 0, 1
_FP8_DTYPES = {FP8_E4M3: "float8_e4m3fn", FP8_E5M2: "float8_e5m2"}


@dataclasses.dataclass
class Fp8Case:
    A: torch.Tensor                # M x K FP8 codes (uint8), CPU
    B: torch.Tensor                # K x N FP8 codes (uint8)
    fmt_a: int
    fmt_b: int
    alpha: float                   # stands in for the product of per-tensor scales
    beta: float
    C0: Optional[torch.Tensor]     # M x N fp32 values, or None


def fp8_codes(x: torch.Tensor, fmt: int) -> torch.Tensor:
    """Round fp32 values to the nearest FP8 value of `fmt` (RNE) and return
    the codes as uint8."""
    return x.to(getattr(torch, _FP8_DTYPES[fmt])).view(torch.uint8).contiguous()


def make_fp8(M: int, N: int, K: int, fmt_a: int = FP8_E4M3, fmt_b: int = FP8_E4M3,
             seed: int = 6, beta: float = 0.0) -> Fp8Case:
    """FP8 GEMM operands: A and B ~ N(0, 1) rounded to FP8, alpha = 1/sqrt(K)
    (the per-tensor scales of a quantised layer fold into alpha, and this one
    keeps C near N(0, 1)); C0 ~ N(0, 1) when beta != 0."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    A = fp8_codes(torch.randn((M, K), generator=gen, dtype=torch.float32), fmt_a)
    B = fp8_codes(torch.randn((K, N), generator=gen, dtype=torch.float32), fmt_b)
    C0 = torch.randn((M, N), generator=gen, dtype=torch.float32) if beta != 0.0 else None
    return Fp8Case(A, B, fmt_a, fmt_b, 1.0 / math.sqrt(max(K, 1)), beta, C0)


@dataclasses.dataclass
class Int4Case:
    q: torch.Tensor                # K x N/2 packed codes (uint8), low nibble = even column
    scales: torch.Tensor           # ceil(K/G) x N bf16
    N: int
    group: int
    zero: int


def pack_int4(codes: torch.Tensor) -> torch.Tensor:
    """K x N codes (0..15, N even) -> K x N/2 bytes, even column in the low nibble."""
    c = codes.to(torch.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).contiguous()


def make_int4(K: int, N: int, group: int = 128, zero: int = 8, seed: int = 8) -> Int4Case:
    """A K x N INT4 weight: codes uniform on 0..15, per-group scales uniform on
    [0.003, 0.006] (with zero point 8 the weights then have the N(0, 0.02)
    spread of the bf16 LLaMA stand-ins), bf16."""
    if N % 2:
        raise ValueError("N must be even (two codes per byte)")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    codes = torch.randint(0, 16, (K, N), generator=gen)
    groups = (K + group - 1) // group
    scales = (0.003 + 0.003 * torch.rand((groups, N), generator=gen)).to(torch.bfloat16)
    return Int4Case(pack_int4(codes), scales, N, group, zero)


@dataclasses.dataclass
class AttentionCase:
    Q: torch.Tensor    # [B][Hq][Sq][D] bf16
    K: torch.Tensor    # [B][Hkv][Sk][D] bf16
    V: torch.Tensor    # [B][Hkv][Sk][D] bf16


def make_attention(B: int = 1, Hq: int = 32, Hkv: int = 32, Sq: int = 2048, Sk: int = 2048,
                   D: int = 128, seed: int = 9) -> AttentionCase:
    """Attention operands, N(0, 1) rounded to bf16; the defaults are one
    LLaMA-7B layer's prefill of a 2048-token context (32 heads of 128)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    Q = torch.randn((B, Hq, Sq, D), generator=gen).to(torch.bfloat16)
    K = torch.randn((B, Hkv, Sk, D), generator=gen).to(torch.bfloat16)
    V = torch.randn((B, Hkv, Sk, D), generator=gen).to(torch.bfloat16)
    return AttentionCase(Q, K, V)
