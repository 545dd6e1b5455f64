"""Run one named GEMM workload through the C ABI a few times (for profiling).

    python -m roofline_driven_optimisation_gb300.run_case --case bf16_8192 --reps 3
    python -m roofline_driven_optimisation_gb300.run_case --case decode_m16_lm --out f32
    python -m roofline_driven_optimisation_gb300.run_case --swiglu 16      (fused FFN gate/up)
    python -m roofline_driven_optimisation_gb300.run_case --fp8 4096       (E4M3 GEMM, n^3)
    python -m roofline_driven_optimisation_gb300.run_case --attention 2048 (32 heads of 128, causal)

Prints the kernel family and the CUDA-event time of each call.  Workload
names are those of ``roofline_driven_optimisation_gb300.inputs``.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch
    import roofline_driven_optimisation_gb300 as g
    from roofline_driven_optimisation_gb300 import inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=sorted(inputs.SPECS))
    ap.add_argument("--swiglu", type=int, metavar="M",
                    help="fused silu(X Wg) * (X Wu) with M rows and the LLaMA-7B gate/up shapes")
    ap.add_argument("--fp8", type=int, metavar="n", help="E4M3 GEMM of size n^3, bf16 C")
    ap.add_argument("--attention", type=int, metavar="S", help="causal attention, 32 heads of 128")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--out", default="auto", choices=["auto", "bf16", "f32"])
    ap.add_argument("--M", type=int)
    ap.add_argument("--N", type=int)
    ap.add_argument("--K", type=int)
    a = ap.parse_args()
    if sum(x is not None for x in (a.case, a.swiglu, a.fp8, a.attention)) != 1:
        ap.error("give exactly one of --case, --swiglu, --fp8 and --attention")

    g.load()
    if a.swiglu is not None:
        return run_swiglu(g, torch, inputs, a)
    if a.fp8 is not None:
        return run_fp8(g, torch, inputs, a)
    if a.attention is not None:
        return run_attention(g, torch, inputs, a)
    c = inputs.make(a.case, M=a.M, N=a.N, K=a.K)
    sp = c.spec
    if sp.in_dtype == "f32":
        out = torch.float32
    else:
        out = torch.float32 if a.out == "f32" else torch.bfloat16
    A, B = c.A.cuda(), c.B.cuda()
    C = c.C0.to(out).cuda() if c.C0 is not None else torch.zeros((sp.M, sp.N), dtype=out, device="cuda")
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gemm(A, B, C, sp.alpha, sp.beta)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"{a.case} M={sp.M} N={sp.N} K={sp.K} path={g.PATH_NAMES[g.last_path()]} "
              f"call {i}: {ms:.4f} ms, {2 * sp.M * sp.N * sp.K / ms / 1e9:.1f} TFLOP/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def run_swiglu(g, torch, inputs, a):
    kw = {k: v for k, v in (("N", a.N), ("K", a.K)) if v is not None}
    c = inputs.make_swiglu(a.swiglu, **kw)
    A, Bg, Bu = c.A.cuda(), c.Bgate.cuda(), c.Bup.cuda()
    M, K = A.shape
    N = Bg.shape[1]
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.swiglu(A, Bg, Bu, C)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        by = 2 * M * K + 4 * K * N + 2 * M * N
        print(f"swiglu M={M} N={N} K={K} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{4 * M * N * K / ms / 1e9:.1f} TFLOP/s, {by / ms / 1e6:.1f} GB/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def run_fp8(g, torch, inputs, a):
    n = a.fp8
    c = inputs.make_fp8(n, n, n, inputs.FP8_E4M3, inputs.FP8_E4M3, seed=7)
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gemm_fp8_tensors(A, 0, B, 0, C, c.alpha)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"fp8 e4m3 n={n} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{2 * n ** 3 / ms / 1e9:.1f} TFLOP/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def run_attention(g, torch, inputs, a):
    S = a.attention
    c = inputs.make_attention(B=1, Hq=32, Hkv=32, Sq=S, Sk=S, D=128, seed=9)
    Q, K, V = c.Q.cuda(), c.K.cuda(), c.V.cuda()
    O = torch.empty_like(Q)
    for i in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.attention(Q, K, V, O, causal=True)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"attention S={S} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{4 * 32 * 128 * S * (S + 1) / 2 / ms / 1e9:.1f} TFLOP/s")
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


if __name__ == "__main__":
    main()
