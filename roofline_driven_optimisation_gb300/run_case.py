"""Run one named GEMM workload through the C ABI a few times (for profiling).

    python -m roofline_driven_optimisation_gb300.run_case --case bf16_8192 --reps 3
    python -m roofline_driven_optimisation_gb300.run_case --case decode_m16_lm --out f32
    python -m roofline_driven_optimisation_gb300.run_case --swiglu 16      (fused FFN gate/up)
    python -m roofline_driven_optimisation_gb300.run_case --fp8 4096       (E4M3 GEMM, n^3)
    python -m roofline_driven_optimisation_gb300.run_case --attention 2048 (32 heads of 128, causal)
    python -m roofline_driven_optimisation_gb300.run_case --attention 4096 --noncausal
    python -m roofline_driven_optimisation_gb300.run_case --int4 16384 --out bf16  (dequantisation, n x n)
    python -m roofline_driven_optimisation_gb300.run_case --w4 16 --N 32000   (INT4-weight decode GEMM)

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
    ap.add_argument("--noncausal", action="store_true", help="attention without the causal mask")
    ap.add_argument("--int4", type=int, metavar="n", help="INT4 dequantisation of an n x n weight (group 128)")
    ap.add_argument("--w4", type=int, metavar="M",
                    help="INT4-weight decode GEMM with M rows (K 4096, N 32000 unless given; group 128)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--out", default="auto", choices=["auto", "bf16", "f32"])
    ap.add_argument("--M", type=int)
    ap.add_argument("--N", type=int)
    ap.add_argument("--K", type=int)
    a = ap.parse_args()
    if sum(x is not None for x in (a.case, a.swiglu, a.fp8, a.attention, a.int4, a.w4)) != 1:
        ap.error("give exactly one of --case, --swiglu, --fp8, --attention, --int4 and --w4")

    g.load()
    if a.swiglu is not None:
        return run_swiglu(g, torch, inputs, a)
    if a.fp8 is not None:
        return run_fp8(g, torch, inputs, a)
    if a.attention is not None:
        return run_attention(g, torch, inputs, a)
    if a.int4 is not None:
        return run_int4(g, torch, inputs, a)
    if a.w4 is not None:
        return run_w4(g, torch, inputs, a)
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


def _report(g):
    status, where = g.device_status()
    if status != 0:
        raise SystemExit(f"device status {status} at site {where}")


def _timed(torch, fn):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def run_attention(g, torch, inputs, a):
    S = a.attention
    causal = not a.noncausal
    c = inputs.make_attention(B=1, Hq=32, Hkv=32, Sq=S, Sk=S, D=128, seed=9)
    Q, K, V = c.Q.cuda(), c.K.cuda(), c.V.cuda()
    O = torch.empty_like(Q)
    pairs = S * (S + 1) // 2 if causal else S * S
    for i in range(a.reps):
        ms = _timed(torch, lambda: g.attention(Q, K, V, O, causal=causal))
        print(f"attention S={S} causal={causal} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{4 * 32 * 128 * pairs / ms / 1e9:.1f} TFLOP/s")
    _report(g)


def run_int4(g, torch, inputs, a):
    n = a.int4
    c = inputs.make_int4(n, n, group=128, zero=8, seed=8)
    q, sc = c.q.cuda(), c.scales.cuda()
    out = torch.float32 if a.out == "f32" else torch.bfloat16
    W = torch.empty((n, n), dtype=out, device="cuda")
    by = q.numel() + sc.numel() * 2 + W.numel() * W.element_size()
    for i in range(a.reps):
        ms = _timed(torch, lambda: g.int4_dequant(q, sc, n, 128, 8, W))
        print(f"int4 dequant n={n} out={a.out} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{by / ms / 1e6:.1f} GB/s")
    _report(g)


def run_w4(g, torch, inputs, a):
    M, K, N = a.w4, a.K or 4096, a.N or 32000
    c = inputs.make_int4(K, N, group=128, zero=8, seed=1)
    qk = g.int4_repack(c.q.cuda(), K, N)
    X = torch.randn((M, K), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).cuda()
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    sc = c.scales.cuda()
    by = K * N // 2 + sc.numel() * 2 + 2 * M * K + 2 * M * N
    for i in range(a.reps):
        ms = _timed(torch, lambda: g.w4a16(X, qk, sc, 128, 8, C))
        print(f"w4a16 M={M} N={N} K={K} path={g.PATH_NAMES[g.last_path()]} call {i}: {ms:.4f} ms, "
              f"{by / ms / 1e6:.1f} GB/s")
    _report(g)


if __name__ == "__main__":
    main()
