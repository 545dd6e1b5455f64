"""FP8 GEMM (E4M3 / E5M2 inputs, bf16 or fp32 C) through the C ABI against the
fp64 oracle on the decoded values.  Error scale: max(|alpha| sum|A||B| +
|beta||C0|) over the decoded operands.  Tolerances: 4e-3 with bf16 C (the
output rounding, 2^-9 relative, dominates); 1e-5 with fp32 C -- the products
of two FP8 values are exact in fp32, so only the fp32 accumulation remains,
as for bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from oracle import fp8
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32
TOL = {BF16: oracle.TOL_BF16_OUT, F32: oracle.TOL_BF16_F32OUT}
E4, E5 = inputs.FP8_E4M3, inputs.FP8_E5M2


def _place(x, pad, off, fill=0):
    rows, cols = x.shape
    ld = max(cols + pad, 1)
    flat = torch.full((off + rows * ld + 16,), fill, dtype=x.dtype)
    flat[off:off + rows * ld].view(rows, ld)[:, :cols] = x
    d = flat.cuda()
    return d, d.data_ptr() + off * d.element_size(), ld


def _run(c, out, *, pad=(0, 0, 0), offset=(0, 0, 0), path=None):
    M, K = c.A.shape
    N = c.B.shape[1]
    A_d, a_ptr, lda = _place(c.A, pad[0], offset[0])
    B_d, b_ptr, ldb = _place(c.B, pad[1], offset[1])
    C_init = c.C0.to(out) if c.C0 is not None else torch.full((M, N), float("nan"), dtype=out)
    C_d, c_ptr, ldc = _place(C_init, pad[2], offset[2], fill=float("nan"))
    fn = g.gemm_fp8 if out == BF16 else g.gemm_fp8_f32out
    if path is not None:
        g.force_path(path)
    try:
        fn(M, N, K, c.alpha, a_ptr, c.fmt_a, lda, b_ptr, c.fmt_b, ldb, c.beta, c_ptr, ldc,
           torch.cuda.current_stream().cuda_stream)
        ran = g.last_path()
    finally:
        g.force_path(g.PATH_AUTO)
    torch.cuda.synchronize()
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"
    full = C_d.cpu()[offset[2]:offset[2] + M * ldc].view(M, ldc)
    return full[:, :N].clone(), ran


def _check(c, out, **kw):
    C, ran = _run(c, out, **kw)
    C0 = c.C0.to(out) if c.C0 is not None else None
    ref = fp8.gemm_fp8(c.A, c.fmt_a, c.B, c.fmt_b, c.alpha, c.beta, C0)
    den = fp8.normwise_denominator_fp8(c.A, c.fmt_a, c.B, c.fmt_b, c.alpha, c.beta, C0)
    err = oracle.normwise_error(C, ref, den if den else 1.0)
    assert err <= TOL[out], f"normwise error {err:.3e} > {TOL[out]:g} (path {g.PATH_NAMES.get(ran)})"
    return err, ran


@pytest.mark.parametrize("out", [BF16, F32])
@pytest.mark.parametrize("fmts", [(E4, E4), (E5, E4), (E4, E5), (E5, E5)])
def test_formats(cuda_lib, out, fmts):
    c = inputs.make_fp8(300, 528, 256, *fmts, seed=sum(fmts) + 1)
    _, ran = _check(c, out)
    assert ran == g.PATH_BF16_TC


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (1, 256, 128), (17, 16, 16), (513, 272, 400),
                                   (1000, 1008, 1040), (256, 4096, 2048), (2048, 512, 64)])
def test_tiles_and_tails(cuda_lib, M, N, K):
    # ragged M, N and K (K = 400: a partial last 128-deep stage; K = 16 and 64:
    # a single partial stage), one and several waves of pair tiles
    c = inputs.make_fp8(M, N, K, E4, E4, seed=M, beta=0.5)
    for out in (BF16, F32):
        _, ran = _check(c, out)
        assert ran == g.PATH_BF16_TC and g.last_tc_pair() in (2, 6)


@pytest.mark.parametrize("M,N,K", [(256, 4096, 2048), (2048, 4096, 1024), (1000, 1008, 1040),
                                   (4096, 4096, 1152)])
def test_fp8_stream_k_tail(cuda_lib, M, N, K):
    # the FP8 pair kernel's tail runs stream-K (it has no half-width tiles):
    # (256, 4096): 16 tiles, all in the tail; (2048, 4096): 52 of 128;
    # (1000, 1008): 9 K-steps of 128 a tile; (4096, 4096): 28 of 256
    c = inputs.make_fp8(M, N, K, E4, E5, seed=K, beta=0.5)
    g.force_split_tiles(2)
    try:
        for out in (BF16, F32):
            _, ran = _check(c, out)
            assert ran == g.PATH_BF16_TC and g.last_tc_pair() == 6, g.last_tc_pair()
        a = _run(c, F32)[0]
        b = _run(c, F32)[0]
        assert torch.equal(a, b)
    finally:
        g.force_split_tiles(1)


def test_fp8_4096_sampled(cuda_lib):
    c = inputs.make_fp8(4096, 4096, 4096, E4, E4, seed=7)
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.empty((4096, 4096), dtype=F32, device="cuda")
    g.gemm_fp8_tensors(A, E4, B, E4, C, c.alpha, 0.0)
    torch.cuda.synchronize()
    assert g.last_path() == g.PATH_BF16_TC
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(4096, 16, replace=False), [0, 4095]]))
    cols = np.unique(np.concatenate([rng.choice(4096, 16, replace=False), [0, 4095]]))
    Cc = C.cpu()
    worst = 0.0
    for A_s, B_s, got in ((c.A[rows], c.B, Cc[rows]), (c.A, c.B[:, cols], Cc[:, cols])):
        ref = fp8.gemm_fp8(A_s, E4, B_s, E4, c.alpha)
        den = fp8.normwise_denominator_fp8(A_s, E4, B_s, E4, c.alpha)
        worst = max(worst, oracle.normwise_error(got, ref, den))
    assert worst <= TOL[F32], worst


@pytest.mark.parametrize("out", [BF16, F32])
def test_generic_kernel(cuda_lib, out):
    c = inputs.make_fp8(70, 90, 52, E5, E4, seed=2, beta=1.5)   # ld not a multiple of 16
    _, ran = _check(c, out)
    assert ran == g.PATH_GENERIC
    c = inputs.make_fp8(64, 128, 64, E4, E5, seed=2)
    _, ran = _check(c, out, path=g.PATH_GENERIC)
    assert ran == g.PATH_GENERIC


def test_padded_and_offset(cuda_lib):
    c = inputs.make_fp8(200, 256, 192, E4, E4, seed=9, beta=0.25)
    _, ran = _check(c, BF16, pad=(16, 32, 5))
    assert ran == g.PATH_BF16_TC
    _, ran = _check(c, F32, offset=(8, 0, 0))   # A 8 bytes off 16-byte alignment
    assert ran == g.PATH_GENERIC


def test_deterministic_and_forced_paths(cuda_lib):
    c = inputs.make_fp8(384, 512, 512, E4, E4, seed=4)
    a1, _ = _run(c, F32)
    a2, _ = _run(c, F32)
    assert torch.equal(a1, a2)
    for path in (g.PATH_F32_SIMT, g.PATH_SKINNY):
        with pytest.raises(g.GemmError) as e:
            _run(c, F32, path=path)
        assert e.value.code == g.GEMM_ERR_UNSUPPORTED


def test_special_values(cuda_lib):
    # a NaN code in A poisons exactly its row of C; K = 0 gives beta*C
    c = inputs.make_fp8(256, 256, 128, E4, E4, seed=5)
    c.A[7, 3] = 0x7F                       # E4M3 NaN
    C, _ = _run(c, F32)
    assert torch.isnan(C[7]).all() and not torch.isnan(C[torch.arange(256) != 7]).any()
    z = inputs.make_fp8(5, 40, 0, E4, E4, seed=1, beta=2.0)
    C, _ = _run(z, F32)
    assert torch.equal(C, 2.0 * z.C0)


def test_bad_format(cuda_lib):
    c = inputs.make_fp8(16, 16, 16)
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.empty((16, 16), dtype=BF16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_fp8(16, 16, 16, 1.0, A.data_ptr(), 2, 16, B.data_ptr(), 0, 16, 0.0, C.data_ptr(), 16, 0)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
