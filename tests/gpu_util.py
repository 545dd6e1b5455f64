"""Helpers shared by the GPU parity tests: run a GEMM through the C ABI and
score it against the CPU oracle with the normwise error."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import roofline_driven_optimisation_gb300 as g

TOL = {("f32", torch.float32): oracle.TOL_F32,
       ("bf16", torch.bfloat16): oracle.TOL_BF16_OUT,
       ("bf16", torch.float32): oracle.TOL_BF16_F32OUT}

FN = {("f32", torch.float32): "gemm_f32",
      ("bf16", torch.bfloat16): "gemm_bf16",
      ("bf16", torch.float32): "gemm_bf16_f32out"}




def run_abi(A_cpu, B_cpu, C0_cpu, alpha, beta, out_dtype, *, pad=(0, 0, 0), offset=(0, 0, 0),
            c_fill=float("nan"), path=None, device="cuda"):
    """Copy operands to the GPU (optionally with padded leading dimensions or
    element offsets from an aligned base), call the C entry point, return C
    (M x N, CPU) and the kernel family that ran."""
    M, K = A_cpu.shape
    N = B_cpu.shape[1]
    in_kind = "f32" if A_cpu.dtype == torch.float32 else "bf16"
    fn = getattr(g, FN[(in_kind, out_dtype)])

    def place(x, extra, off, fill):
        rows, cols = x.shape
        ld = cols + extra
        flat = torch.full((off + rows * ld + 8,), fill, dtype=x.dtype)
        view = flat[off:off + rows * ld].view(rows, ld)
        view[:, :cols] = x
        return flat.to(device), max(ld, 1)

    A_d, lda = place(A_cpu, pad[0], offset[0], 0.0)
    B_d, ldb = place(B_cpu, pad[1], offset[1], 0.0)
    C_init = C0_cpu.to(out_dtype) if C0_cpu is not None else torch.full((M, N), c_fill, dtype=out_dtype)
    C_d, ldc = place(C_init, pad[2], offset[2], c_fill)
    esz_in = A_cpu.element_size()
    esz_out = torch.empty((), dtype=out_dtype).element_size()
    a_ptr = A_d.data_ptr() + offset[0] * esz_in
    b_ptr = B_d.data_ptr() + offset[1] * esz_in
    c_ptr = C_d.data_ptr() + offset[2] * esz_out
    s = torch.cuda.current_stream().cuda_stream
    if path is not None:
        g.force_path(path)
    try:
        fn(M, N, K, float(alpha), a_ptr, lda, b_ptr, ldb, float(beta), c_ptr, ldc, s)
        ran = g.last_path()
    finally:
        if path is not None:
            g.force_path(g.PATH_AUTO)
    torch.cuda.synchronize()
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"
    C_full = C_d.cpu()[offset[2]:offset[2] + M * ldc].view(M, ldc)
    return C_full[:, :N].clone(), C_full[:, N:].clone(), ran


def check(A_cpu, B_cpu, C0_cpu, alpha, beta, out_dtype, *, tol=None, strict=None, **kw):
    """Run through the ABI, score against the oracle; returns (err, path).

    The scale is that of the whole expression (|alpha||A||B| + |beta||C0|);
    strict=True also requires the bound with the plain max sum_k |A||B|.  By
    default every case is strict except bf16 C with beta != 0, whose rounding
    is relative to |beta*C0| as well (at small K no correctly rounded result
    meets the bound against sum |A||B| alone)."""
    in_kind = "f32" if A_cpu.dtype == torch.float32 else "bf16"
    tol = TOL[(in_kind, out_dtype)] if tol is None else tol
    if strict is None:
        strict = not (out_dtype == torch.bfloat16 and beta != 0.0)
    C, pad_cols, ran = run_abi(A_cpu, B_cpu, C0_cpu, alpha, beta, out_dtype, **kw)
    C0_exact = C0_cpu.to(out_dtype) if C0_cpu is not None else None
    ref = oracle.gemm(A_cpu, B_cpu, alpha, beta, C0_exact)
    denom = oracle.normwise_denominator(A_cpu, B_cpu, alpha, beta, C0_exact)
    if denom == 0.0:
        denom = 1.0
    err = oracle.normwise_error(C, ref, denom)
    assert err <= tol, f"normwise error {err:.3e} > {tol:g} (path {g.PATH_NAMES.get(ran)})"
    if strict:
        plain = oracle.abs_product_max(A_cpu, B_cpu)
        err_plain = oracle.normwise_error(C, ref, plain if plain else 1.0)
        assert err_plain <= tol, f"normwise error (plain scale) {err_plain:.3e} > {tol:g}"
    # the padding of C's rows is never written
    if pad_cols.numel():
        pc = pad_cols.to(torch.float64).numpy()
        assert np.all(np.isnan(pc)) or np.all(pc == pc.flat[0])
    return err, ran


def sampled_check(A_dev, B_dev, C_dev, A_cpu, B_cpu, C0_cpu, alpha, beta, tol, rows, cols,
                  *, strict=False):
    """Full-size check on sampled rows and columns (the oracle computes each
    sampled row or column exactly); the denominator is the max over the sample.

    The scale is that of the whole expression (|alpha||A||B| + |beta||C0|);
    strict=True also requires the bound with the plain max sum_k |A||B| over
    the sample, the normwise error as the GEMM's definition states it."""
    C_cpu = C_dev.cpu()
    worst = worst_plain = 0.0
    for sel_rows in (True, False):
        if sel_rows:
            A_s, B_s = A_cpu[rows], B_cpu
            G = C_cpu[rows]
            C0_s = C0_cpu[rows] if C0_cpu is not None else None
        else:
            A_s, B_s = A_cpu, B_cpu[:, cols]
            G = C_cpu[:, cols]
            C0_s = C0_cpu[:, cols] if C0_cpu is not None else None
        ref = oracle.gemm(A_s, B_s, alpha, beta, C0_s)
        denom = oracle.normwise_denominator(A_s, B_s, alpha, beta, C0_s)
        err = oracle.normwise_error(G, ref, denom if denom else 1.0)
        worst = max(worst, err)
        if strict:
            plain = oracle.abs_product_max(A_s, B_s)
            worst_plain = max(worst_plain, oracle.normwise_error(G, ref, plain if plain else 1.0))
    assert worst <= tol, f"sampled normwise error {worst:.3e} > {tol:g}"
    if strict:
        assert worst_plain <= tol, f"sampled normwise error (plain scale) {worst_plain:.3e} > {tol:g}"
    return max(worst, worst_plain)
