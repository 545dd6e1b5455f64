"""GPU parity: every kernel family against the CPU oracle, through the C ABI.

Sizes the oracle finishes in seconds still span several tiles and a ragged
tail; full-size workloads are checked on sampled rows and columns.  Scores are
the normwise error max|C_gpu - C_ref| / max(sum_k |A||B|) with the bounds
1e-5 (fp32 path), 4e-3 (bf16 inputs, bf16 C), 1e-5 (bf16 inputs, fp32 C).
"""
import numpy as np
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from roofline_driven_optimisation_gb300 import inputs
from gpu_util import check, run_abi, sampled_check

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


def expected_path(M, N, K, in_kind):
    """Kernel family the dispatcher must pick for packed row-major operands:
    TMA needs leading dimensions whose byte size is a multiple of 16."""
    per16 = 4 if in_kind == "f32" else 8
    if K == 0 or K % per16 or N % per16:
        return g.PATH_GENERIC
    if in_kind == "f32":
        return g.PATH_F32_SIMT
    return g.PATH_SKINNY if M <= 16 else g.PATH_BF16_TC


# ------------------------------------------------------------------ fp32 path
def test_fp32_256_full(cuda_lib):
    c = inputs.make("fp32_256")
    err, path = check(c.A, c.B, None, 1.0, 0.0, F32, strict=True)
    assert path == g.PATH_F32_SIMT


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 9, 5), (129, 257, 33), (129, 260, 36),
                                   (300, 200, 1000), (513, 388, 96), (64, 4100, 20), (1, 132, 4)])
def test_fp32_ragged(cuda_lib, M, N, K):
    c = inputs.make("fp32_4096", M=M, N=N, K=K)
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32)
    assert path == expected_path(M, N, K, "f32")


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K", [(7, 12, 16), (129, 260, 36), (128, 256, 16), (255, 516, 200),
                                   (300, 1000, 332), (513, 388, 96), (64, 4100, 20)])
def test_fp32_each_tile_width(cuda_lib, bn, M, N, K):
    # 128: 8 x 8 register tiles on 128 x 128 C tiles, two CTAs per SM;
    # 256: 8 x 16 register tiles on 128 x 256 C tiles, one CTA per SM
    c = inputs.make("fp32_4096", M=M, N=N, K=K)
    g.force_tile_n(bn)
    try:
        err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32)
        assert path == g.PATH_F32_SIMT and g.last_tile_n() == bn
        err, path = check(c.A, c.B, None, 1.0, 0.0, F32, c_fill=float("nan"))
        assert g.last_tile_n() == bn
    finally:
        g.force_tile_n(0)


def test_fp32_forced_widths_other_than_128_and_256_are_refused(cuda_lib):
    c = inputs.make("fp32_4096", M=64, N=64, K=16)
    g.force_tile_n(192)
    try:
        with pytest.raises(g.GemmError) as e:
            run_abi(c.A, c.B, None, 1.0, 0.0, F32)
        assert e.value.code == g.GEMM_ERR_UNSUPPORTED
    finally:
        g.force_tile_n(0)


@pytest.mark.parametrize("alpha,beta", [(0.0, 0.0), (1.0, 0.0), (-1.0, 0.5), (1.5, 1.0), (1.0, 0.5)])
def test_fp32_alpha_beta_grid(cuda_lib, alpha, beta):
    c = inputs.make("fp32_4096", M=200, N=160, K=64)
    check(c.A, c.B, c.C0, alpha, beta, F32)


def test_fp32_beta_zero_ignores_nan_c(cuda_lib):
    c = inputs.make("fp32_256", M=130, N=140, K=40)
    C, _, _ = run_abi(c.A, c.B, None, 1.0, 0.0, F32, c_fill=float("nan"))
    assert torch.isfinite(C).all()


def test_fp32_padded_leading_dims(cuda_lib):
    c = inputs.make("fp32_4096", M=150, N=260, K=72)
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, pad=(4, 8, 12))
    assert path == g.PATH_F32_SIMT


def test_fp32_misaligned_runs_generic(cuda_lib):
    c = inputs.make("fp32_4096", M=70, N=92, K=52)
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32)
    assert path == g.PATH_F32_SIMT
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, offset=(1, 0, 0))
    assert path == g.PATH_GENERIC
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, pad=(1, 0, 0))   # lda*4 not a multiple of 16
    assert path == g.PATH_GENERIC


def test_fp32_unaligned_c_uses_scalar_epilogue(cuda_lib):
    c = inputs.make("fp32_4096", M=140, N=132, K=40)
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, offset=(0, 0, 1), pad=(0, 0, 3))
    assert path == g.PATH_F32_SIMT


def test_fp32_k_zero(cuda_lib):
    c = inputs.make("fp32_4096", M=33, N=45, K=1)
    A = c.A[:, :0].contiguous()
    B = c.B[:0, :].contiguous()
    C, _, path = run_abi(A, B, c.C0, 1.5, 0.5, F32)
    assert path == g.PATH_GENERIC
    assert torch.equal(C, 0.5 * c.C0)


def test_fp32_forced_generic_matches_oracle(cuda_lib):
    c = inputs.make("fp32_4096", M=190, N=170, K=150)
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, path=g.PATH_GENERIC)
    assert path == g.PATH_GENERIC


@pytest.mark.parametrize("bn", [0, 128, 256])
def test_fp32_4096_full_size_sampled(cuda_lib, bn):
    # bn 0: the dispatcher's choice (the bench's launch configuration)
    c = inputs.make("fp32_4096")
    A, B, C = c.A.cuda(), c.B.cuda(), c.C0.cuda()
    g.force_tile_n(bn)
    try:
        g.gemm(A, B, C, 1.5, 0.5)
        torch.cuda.synchronize()
    finally:
        g.force_tile_n(0)
    assert g.last_path() == g.PATH_F32_SIMT
    assert bn == 0 or g.last_tile_n() == bn
    # 128-wide: 1024 tiles = 3 waves of 304 + 112; 256-wide: 512 tiles = 3
    # waves of 152 + 56; whether the rest splits depends on how many clusters
    # fit at once
    assert g.last_k_split() in (1, 2, 4)
    gen = np.random.default_rng(11)
    rows = np.sort(gen.choice(4096, 24, replace=False))
    cols = np.sort(gen.choice(4096, 24, replace=False))
    sampled_check(A, B, C, c.A, c.B, c.C0, 1.5, 0.5, oracle.TOL_F32, rows, cols, strict=True)


# The splits each width takes for these shapes on GB300 (152 SMs): 128-wide
# tiles split four ways (at least 64 clusters of four fit at once); 256-wide
# tiles run their last partial wave stream-K, and last_k_split() reports how
# many CTAs shared the most-shared tile (two or more here).


def _expect_split(bn, split):
    return split == 4 if bn == 128 else split >= 2


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K,pad", [(1024, 1024, 1024, (0, 0, 0)), (2560, 2048, 1024, (0, 0, 0)),
                                       (1000, 1004, 1001, (3, 0, 0)), (300, 200, 1000, (0, 0, 0))])
def test_fp32_split_last_wave(cuda_lib, bn, M, N, K, pad):
    # 128-wide: 1024^2: 64 tiles, all in the split launch; 2560 x 2048: 320
    # tiles, the 16 past two whole waves of 2 x 152 split; 1000 x 1004 x 1001:
    # ragged M, N and K (63 K-slices, ranks take 15/16/16/16); 300 x 200: six
    # tiles.  256-wide: 32, 160 (8 past one wave of 152), 32 and 3 tiles, the
    # tiles past the last whole wave stream-K over the SMs.
    c = inputs.make("fp32_4096", M=M, N=N, K=K)
    g.force_tile_n(bn)
    try:
        err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, pad=pad)
        assert path == g.PATH_F32_SIMT and _expect_split(bn, g.last_k_split())
        # partial sums are added in rank order: repeated calls give the same bits
        a = run_abi(c.A, c.B, c.C0, 1.5, 0.5, F32, pad=pad)[0]
        b = run_abi(c.A, c.B, c.C0, 1.5, 0.5, F32, pad=pad)[0]
        assert torch.equal(a, b)
        g.force_split_tiles(0)
        try:
            check(c.A, c.B, c.C0, 1.5, 0.5, F32, pad=pad)
            assert g.last_k_split() == 1
        finally:
            g.force_split_tiles(1)
    finally:
        g.force_tile_n(0)


@pytest.mark.parametrize("N", [1024, 1000, 900, 800])
def test_fp32_wide_tiles_ragged_n_split(cuda_lib, N):
    # 256-wide tiles with the last column of tiles partly outside C (N = 1000,
    # 900: the right half holds 232 or 132 columns; 800: 32), every tile in
    # the split launch (2048 x N: 16 x 4 tiles, fewer than one wave of 152)
    c = inputs.make("fp32_4096", M=2048, N=N, K=1024)
    g.force_tile_n(256)
    try:
        err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32)
        assert path == g.PATH_F32_SIMT and g.last_tile_n() == 256 and g.last_k_split() in (2, 4)
        err, path = check(c.A, c.B, None, 1.0, 0.0, F32, c_fill=float("nan"), pad=(0, 0, 4))
    finally:
        g.force_tile_n(0)


def test_fp32_4096_configuration(cuda_lib):
    # the bench's shape at a shorter K: on 152 SMs the wave model picks the
    # 256-wide tiles (512 tiles = 3 waves of 152 + 56, the 56 tiles' 56 x 64
    # K-slices stream-K over 152 CTAs of 23-24 slices: a tile meets 3-4 CTAs)
    c = inputs.make("fp32_4096", M=4096, N=4096, K=1024)
    check(c.A, c.B, c.C0, 1.5, 0.5, F32)
    assert g.last_path() == g.PATH_F32_SIMT
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert g.last_tile_n() == 256 and g.last_k_split() in (3, 4)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256),      # one tile, one CTA: no partner
                                   (4096, 4096, 256),    # 56 tiles over 56 CTAs, one tile each
                                   (1536, 2560, 776),    # 12 x 10 tiles, ragged K (49 slices)
                                   (300, 520, 4096),     # 3 x 3 tiles over 152 CTAs
                                   (2048, 2048, 4096),   # 128 tiles, no whole wave
                                   (4224, 4352, 640)])   # 33 x 17 = 561 tiles: 3 waves + 105
def test_fp32_stream_k_tail(cuda_lib, M, N, K):
    # the 256-wide tiles' last partial wave as stream-K: K-slice ranges that
    # start and end inside tiles, partial tiles meeting in the workspace; the
    # finisher adds them in a fixed order, so four calls in a row (each on
    # the next of the four workspace slots) give the same bits
    c = inputs.make("fp32_4096", M=M, N=N, K=K)
    g.force_tile_n(256)
    try:
        err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32)
        assert path == g.PATH_F32_SIMT and g.last_tile_n() == 256
        outs = [run_abi(c.A, c.B, c.C0, 1.5, 0.5, F32)[0] for _ in range(4)]
        assert all(torch.equal(outs[0], o) for o in outs[1:])
        err, path = check(c.A, c.B, None, 1.0, 0.0, F32, c_fill=float("nan"), offset=(0, 0, 1), pad=(0, 0, 3))
    finally:
        g.force_tile_n(0)


@pytest.mark.parametrize("bn", [128, 256])
def test_fp32_split_unaligned_c_and_nan_c(cuda_lib, bn):
    # the split epilogue's scalar path (C one element past an aligned base,
    # ldc not a multiple of 4), and beta = 0 over a NaN-filled C
    c = inputs.make("fp32_4096", M=300, N=200, K=1000)
    g.force_tile_n(bn)
    try:
        err, path = check(c.A, c.B, c.C0, 1.5, 0.5, F32, offset=(0, 0, 1), pad=(0, 0, 3))
        assert path == g.PATH_F32_SIMT and _expect_split(bn, g.last_k_split())
        C, _, _ = run_abi(c.A, c.B, None, 1.0, 0.0, F32, c_fill=float("nan"))
        assert _expect_split(bn, g.last_k_split()) and torch.isfinite(C).all()
    finally:
        g.force_tile_n(0)


@pytest.mark.parametrize("bn", [128, 256])
def test_fp32_split_result_feeds_next_call(cuda_lib, bn):
    # the split launch overlaps the end of the whole-wave launch; a GEMM queued
    # right after must still read every tile of C1 final (C1 starts as NaN)
    c = inputs.make("fp32_4096", M=2560, N=2048, K=1024)
    D_cpu = inputs.make("fp32_4096", M=1, N=512, K=2048).B
    A, B, D = c.A.cuda(), c.B.cuda(), D_cpu.cuda()
    C1 = torch.empty(2560, 2048, device="cuda")
    C2 = torch.empty(2560, 512, device="cuda")
    for _ in range(3):
        C1.fill_(float("nan"))
        g.force_tile_n(bn)
        try:
            g.gemm(A, B, C1, 1.0, 0.0)
            assert _expect_split(bn, g.last_k_split())
        finally:
            g.force_tile_n(0)
        g.gemm(C1, D, C2, 1.0, 0.0)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    C1_cpu = C1.cpu()
    assert torch.isfinite(C1_cpu).all() and torch.isfinite(C2.cpu()).all()
    ref = oracle.gemm(C1_cpu, D_cpu, 1.0, 0.0, None)
    denom = oracle.normwise_denominator(C1_cpu, D_cpu, 1.0, 0.0, None)
    assert oracle.normwise_error(C2.cpu(), ref, denom) <= oracle.TOL_F32


# ------------------------------------------------------------------ bf16 tensor-core path
@pytest.mark.parametrize("out", [BF16, F32])
@pytest.mark.parametrize("M,N,K", [(17, 8, 64), (128, 256, 64), (256, 512, 320), (300, 520, 200),
                                   (129, 296, 1000), (640, 264, 72), (1000, 1000, 1000),
                                   (33, 300, 100), (260, 136, 8)])
def test_bf16_tc_ragged(cuda_lib, M, N, K, out):
    c = inputs.make("bf16_4096", M=M, N=N, K=K)
    err, path = check(c.A, c.B, None, 1.0, 0.0, out)
    assert path == expected_path(M, N, K, "bf16")


@pytest.mark.parametrize("out", [BF16, F32])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.0, 0.5), (-1.0, 1.0), (1.5, 0.5)])
def test_bf16_tc_alpha_beta(cuda_lib, out, alpha, beta):
    c = inputs.make("decode_m16_o", M=200, N=384, K=256)   # normal C0 for the beta term
    err, path = check(c.A, c.B, c.C0, alpha, beta, out)
    assert path == g.PATH_BF16_TC


@pytest.mark.parametrize("bn", [128, 192, 224, 256])
@pytest.mark.parametrize("M,N,K", [(300, 1000, 200), (256, 4096, 128), (140, 456, 520)])
def test_bf16_tc_every_tile_width(cuda_lib, bn, M, N, K):
    c = inputs.make("decode_m16_o", M=M, N=N, K=K)
    g.force_tile_n(bn)
    g.force_tc_pair(1)
    try:
        for out, beta in ((BF16, 0.0), (F32, 0.5)):
            err, path = check(c.A, c.B, c.C0, 1.0, beta, out)
            assert path == g.PATH_BF16_TC and g.last_tile_n() == bn and g.last_tc_pair() == 1
    finally:
        g.force_tile_n(0)
        g.force_tc_pair(0)


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("M,N,K", [(17, 64, 64), (100, 304, 136), (256, 256, 64), (300, 1000, 200),
                                   (520, 640, 1000), (1024, 2048, 256)])
def test_bf16_tc_pair(cuda_lib, bn, M, N, K):
    c = inputs.make("decode_m16_o", M=M, N=N, K=K)
    g.force_tc_pair(2)
    g.force_tile_n(bn)
    try:
        for out, alpha, beta in ((BF16, 1.0, 0.0), (F32, 1.5, 0.5)):
            err, path = check(c.A, c.B, c.C0, alpha, beta, out)
            assert path == g.PATH_BF16_TC and g.last_tc_pair() in (2, 4, 6) and g.last_tile_n() == bn
    finally:
        g.force_tc_pair(0)
        g.force_tile_n(0)


def test_bf16_tc_pair_deterministic_and_matches_single(cuda_lib):
    c = inputs.make("bf16_4096", M=768, N=1024, K=512)
    g.force_tc_pair(2)
    try:
        a = run_abi(c.A, c.B, None, 1.0, 0.0, F32)[0]
        b = run_abi(c.A, c.B, None, 1.0, 0.0, F32)[0]
    finally:
        g.force_tc_pair(0)
    assert torch.equal(a, b)
    g.force_tc_pair(1)
    try:
        s1 = run_abi(c.A, c.B, None, 1.0, 0.0, F32)[0]
    finally:
        g.force_tc_pair(0)
    # same products, same k order inside each 16-deep MMA step: agree to fp32 rounding
    assert torch.allclose(a, s1, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("M,N,K", [(2560, 2560, 1024), (1536, 1280, 1024), (1300, 1000, 520),
                                   (1300, 800, 520), (300, 256, 136)])
def test_bf16_tc_half_width_last_wave(cuda_lib, M, N, K):
    # tile counts whose partial last wave runs as half-width tiles; (1300, 800):
    # the second half of the last tile column lies entirely outside C;
    # (1536, 1280) and (300, 256): fewer tiles than pairs, every tile halved
    c = inputs.make("decode_m16_o", M=M, N=N, K=K)
    g.force_tc_pair(2)
    g.force_tile_n(256)
    g.force_split_tiles(3)   # pin the half-width tail
    try:
        for out, alpha, beta in ((BF16, 1.0, 0.0), (F32, 1.5, 0.5)):
            err, path = check(c.A, c.B, c.C0, alpha, beta, out)
            assert path == g.PATH_BF16_TC and g.last_tc_pair() == 4, g.last_tc_pair()
        a1 = run_abi(c.A, c.B, None, 1.0, 0.0, F32)[0]
        g.force_split_tiles(0)
        b = run_abi(c.A, c.B, None, 1.0, 0.0, F32)[0]
        assert g.last_tc_pair() == 2
        # the same products in the same order: identical bits
        assert torch.equal(a1, b)
    finally:
        g.force_split_tiles(1)
        g.force_tc_pair(0)
        g.force_tile_n(0)


@pytest.mark.parametrize("M,N,K", [(2560, 2560, 1024), (1536, 1280, 1024), (1300, 1000, 520),
                                   (2048, 4096, 768), (300, 520, 4096), (1000, 1008, 1000)])
def test_bf16_tc_stream_k_tail(cuda_lib, M, N, K):
    # the tiles past the last whole wave of pairs run stream-K: their K-steps
    # spread evenly over the pairs, partial tiles added by each tile's
    # finisher in pair order.  (2560, 2560): 100 tiles, 24 in the tail;
    # (1536, 1280), (300, 520), (1000, 1008): fewer tiles than pairs, all in
    # the tail; (1300, 1000): 9 K-steps a tile; (2048, 4096): 52 tail tiles
    # of 12 K-steps over every pair, up to three pairs meeting in a tile
    c = inputs.make("decode_m16_o", M=M, N=N, K=K)
    g.force_tc_pair(2)
    g.force_tile_n(256)
    g.force_split_tiles(2)   # pin the stream-K tail
    try:
        for out, alpha, beta in ((BF16, 1.0, 0.0), (F32, 1.5, 0.5)):
            err, path = check(c.A, c.B, c.C0, alpha, beta, out)
            assert path == g.PATH_BF16_TC and g.last_tc_pair() == 6, g.last_tc_pair()
        # the addition order depends on the shape alone: identical bits on
        # every call (five calls: every workspace slot is used)
        first = run_abi(c.A, c.B, c.C0, 1.5, 0.5, F32)[0]
        for _ in range(4):
            assert torch.equal(run_abi(c.A, c.B, c.C0, 1.5, 0.5, F32)[0], first)
        g.force_split_tiles(0)
        whole = run_abi(c.A, c.B, c.C0, 1.5, 0.5, F32)[0]
        assert g.last_tc_pair() == 2
        # another fp32 summation order of the same products: the same bound
        den = oracle.normwise_denominator(c.A, c.B, 1.5, 0.5, c.C0.to(F32))
        assert oracle.normwise_error(first, oracle.to_f64(whole), den) <= oracle.TOL_BF16_F32OUT
    finally:
        g.force_split_tiles(1)
        g.force_tc_pair(0)
        g.force_tile_n(0)


def test_bf16_tc_pair_rejects_other_widths(cuda_lib):
    c = inputs.make("bf16_4096", M=256, N=256, K=64)
    g.force_tc_pair(2)
    g.force_tile_n(192)
    try:
        with pytest.raises(g.GemmError) as e:
            run_abi(c.A, c.B, None, 1.0, 0.0, BF16)
        assert e.value.code == g.GEMM_ERR_UNSUPPORTED
    finally:
        g.force_tc_pair(0)
        g.force_tile_n(0)
    with pytest.raises(g.GemmError):
        g.force_tc_pair(3)


@pytest.mark.parametrize("out", [BF16, F32])
def test_bf16_tc_pair_8192_sampled(cuda_lib, out):
    c = inputs.make("bf16_8192")
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.full((8192, 8192), float("nan"), dtype=out, device="cuda")
    g.force_tc_pair(2)
    try:
        g.gemm(A, B, C, 1.0, 0.0)
        torch.cuda.synchronize()
        assert g.last_tc_pair() in (2, 4, 6)
    finally:
        g.force_tc_pair(0)
    gen = np.random.default_rng(7)
    rows = np.sort(gen.choice(8192, 12, replace=False))
    cols = np.sort(gen.choice(8192, 12, replace=False))
    tol = oracle.TOL_BF16_OUT if out == BF16 else oracle.TOL_BF16_F32OUT
    sampled_check(A, B, C, c.A, c.B, None, 1.0, 0.0, tol, rows, cols, strict=True)


def test_bf16_tc_tile_width_choice(cuda_lib):
    # on 152 SMs: square 4096 and 8192 run on CTA pairs with 256 x 256 tiles
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, N, want in ((8192, 8192, (2, 256)), (4096, 4096, (2, 256))):
        c = inputs.make("bf16_4096", M=M, N=N, K=64)
        check(c.A, c.B, None, 1.0, 0.0, BF16)
        if sms == 152:
            assert (min(g.last_tc_pair(), 2), g.last_tile_n()) == want, (M, N)
    with pytest.raises(g.GemmError):
        g.force_tile_n(100)


def test_bf16_dispatcher_counts_the_halved_last_wave(cuda_lib):
    # 512 x 11008: 86 pair tiles of 256 x 256 = one wave of 76 pairs and 10
    # tiles halved on 20 pairs, which beats single-CTA 192-wide tiles on
    # GB300 (47.1 against 52.0 us at K = 4096); with the split forbidden the
    # dispatcher keeps the single-CTA tiles
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    c = inputs.make("bf16_4096", M=512, N=11008, K=256)
    for out in (BF16, F32):
        check(c.A, c.B, None, 1.0, 0.0, out)
        if sms == 152:
            assert (g.last_tc_pair(), g.last_tile_n()) == (4, 256)
    g.force_split_tiles(0)
    try:
        check(c.A, c.B, None, 1.0, 0.0, BF16)
        if sms == 152:
            assert (g.last_tc_pair(), g.last_tile_n()) == (1, 192)
    finally:
        g.force_split_tiles(1)


def test_bf16_tc_padded_and_unaligned_c(cuda_lib):
    c = inputs.make("bf16_4096", M=260, N=272, K=136)
    check(c.A, c.B, None, 1.0, 0.0, BF16, pad=(8, 16, 3))
    err, path = check(c.A, c.B, None, 1.0, 0.0, BF16, offset=(0, 0, 1))
    assert path == g.PATH_BF16_TC
    err, path = check(c.A, c.B, None, 1.0, 0.0, F32, offset=(0, 0, 1), pad=(0, 0, 1))
    assert path == g.PATH_BF16_TC


def test_bf16_misaligned_runs_generic(cuda_lib):
    c = inputs.make("bf16_4096", M=100, N=120, K=88)
    for kw in (dict(offset=(1, 0, 0)), dict(offset=(0, 3, 0)), dict(pad=(2, 0, 0)), dict(pad=(0, 1, 0))):
        err, path = check(c.A, c.B, None, 1.0, 0.0, BF16, **kw)
        assert path == g.PATH_GENERIC, kw
    err, path = check(c.A, c.B, None, 1.0, 0.0, F32, offset=(1, 0, 0))
    assert path == g.PATH_GENERIC


def test_bf16_deterministic(cuda_lib):
    c = inputs.make("bf16_4096", M=512, N=768, K=640)
    outs = [run_abi(c.A, c.B, None, 1.0, 0.0, F32)[0] for _ in range(2)]
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("n", [4096, 8192])
@pytest.mark.parametrize("out", [BF16, F32])
def test_bf16_square_full_size_sampled(cuda_lib, n, out):
    c = inputs.make(f"bf16_{n}")
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.full((n, n), float("nan"), dtype=out, device="cuda")
    g.gemm(A, B, C, 1.0, 0.0)
    torch.cuda.synchronize()
    assert g.last_path() == g.PATH_BF16_TC
    gen = np.random.default_rng(n)
    rows = np.sort(gen.choice(n, 16, replace=False))
    cols = np.sort(gen.choice(n, 16, replace=False))
    tol = oracle.TOL_BF16_OUT if out == BF16 else oracle.TOL_BF16_F32OUT
    sampled_check(A, B, C, c.A, c.B, None, 1.0, 0.0, tol, rows, cols, strict=True)


@pytest.mark.parametrize("w", ["qkv", "o", "gate", "down", "lm"])
def test_prefill_full_size_sampled(cuda_lib, w):
    c = inputs.make(f"prefill_{w}")
    A, B = c.A.cuda(), c.B.cuda()
    C = torch.empty((c.spec.M, c.spec.N), dtype=BF16, device="cuda")
    g.gemm(A, B, C, 1.0, 0.0)
    torch.cuda.synchronize()
    gen = np.random.default_rng(3)
    rows = np.sort(gen.choice(c.spec.M, 8, replace=False))
    cols = np.sort(gen.choice(c.spec.N, 8, replace=False))
    sampled_check(A, B, C, c.A, c.B, None, 1.0, 0.0, oracle.TOL_BF16_OUT, rows, cols,
                  strict=True)


# ------------------------------------------------------------------ skinny split-K path
@pytest.mark.parametrize("m", [1, 4, 16])
@pytest.mark.parametrize("N,K", [(384, 512), (4104, 1000), (200, 64), (96, 11008), (1000, 72), (8, 8)])
def test_skinny_ragged(cuda_lib, m, N, K):
    c = inputs.make(f"decode_m{m}_o", M=m, N=N, K=K)
    for out in (BF16, F32):
        err, path = check(c.A, c.B, c.C0, 1.0, 1.0, out)
        assert path == g.PATH_SKINNY


@pytest.mark.parametrize("m", [2, 3, 5, 9, 15])
def test_skinny_odd_m(cuda_lib, m):
    c = inputs.make("decode_m16_o", M=m, N=520, K=392)
    err, path = check(c.A, c.B, c.C0, 1.5, 0.5, BF16, pad=(8, 8, 5))
    assert path == g.PATH_SKINNY


@pytest.mark.parametrize("m", [1, 4, 16])
@pytest.mark.parametrize("w", ["qkv", "o", "gate", "down", "lm"])
def test_decode_full_size(cuda_lib, m, w):
    # decode GEMMs are small enough for the oracle to check every element
    c = inputs.make(f"decode_m{m}_{w}")
    err, path = check(c.A, c.B, c.C0, 1.0, 1.0, BF16, strict=True)
    assert path == g.PATH_SKINNY


def test_skinny_deterministic_and_split_consistent(cuda_lib):
    c = inputs.make("decode_m16_down", K=4096, N=1024)
    a = run_abi(c.A, c.B, c.C0, 1.0, 1.0, F32)[0]
    b = run_abi(c.A, c.B, c.C0, 1.0, 1.0, F32)[0]
    assert torch.equal(a, b)


def test_forced_paths_agree(cuda_lib):
    c = inputs.make("decode_m16_o", M=16, N=640, K=512)
    e1, p1 = check(c.A, c.B, c.C0, 1.0, 1.0, F32, path=g.PATH_SKINNY)
    e2, p2 = check(c.A, c.B, c.C0, 1.0, 1.0, F32, path=g.PATH_BF16_TC)
    e3, p3 = check(c.A, c.B, c.C0, 1.0, 1.0, F32, path=g.PATH_GENERIC)
    assert (p1, p2, p3) == (g.PATH_SKINNY, g.PATH_BF16_TC, g.PATH_GENERIC)


def test_forced_path_rejects_wrong_family(cuda_lib):
    c = inputs.make("decode_m16_o", M=32, N=64, K=64)
    with pytest.raises(g.GemmError) as e:
        run_abi(c.A, c.B, c.C0, 1.0, 1.0, BF16, path=g.PATH_SKINNY)   # M > 16
    assert e.value.code == g.GEMM_ERR_UNSUPPORTED
    f = inputs.make("fp32_256", M=16, N=16, K=16)
    with pytest.raises(g.GemmError) as e:
        run_abi(f.A, f.B, None, 1.0, 0.0, F32, path=g.PATH_BF16_TC)
    assert e.value.code == g.GEMM_ERR_UNSUPPORTED


# ------------------------------------------------------------------ status and errors
def test_bounded_wait_reports_timeout(cuda_lib):
    assert g.device_status()[0] == 0
    g.selftest_wait_timeout(2_000_000)   # 2 ms on a barrier nothing arrives at
    status, where = g.device_status()
    assert status == g.GEMM_ERR_DEVICE_TIMEOUT and where == 1
    assert g.device_status()[0] == 0      # read-and-clear
    # the context is still usable
    c = inputs.make("fp32_256", M=64, N=64, K=64)
    check(c.A, c.B, None, 1.0, 0.0, F32)


def test_invalid_arguments(cuda_lib):
    x = torch.zeros(1024, device="cuda")
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32(4, 4, 8, 1.0, p, 4, p, 4, 0.0, p, 4, s)     # lda < K
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32(4, 4, 4, 1.0, 0, 4, p, 4, 0.0, p, 4, s)     # null A
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32(4, 4, 4, 1.0, p + 2, 4, p, 4, 0.0, p, 4, s)  # not float-aligned
    assert e.value.code == g.GEMM_ERR_MISALIGNED
    g.gemm_f32(0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4, s)         # no-op
    assert g.last_path() == g.PATH_AUTO


def test_many_distinct_operands(cuda_lib):
    # more distinct (pointer, shape) operands than the per-thread tensor-map
    # cache holds: the cache empties between calls, never inside one, so a
    # call's first map stays valid while its second is made
    M = N = K = 64
    gen = torch.Generator().manual_seed(41)
    A_all = torch.randn((700 * 8 + M * K,), generator=gen).to(BF16)
    B_all = torch.randn((700 * 8 + K * N,), generator=gen).to(BF16)
    A_d, B_d = A_all.cuda(), B_all.cuda()
    C = torch.zeros((M, N), dtype=F32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for i in range(700):
        off = 8 * i   # 16-byte steps: every call gets new A and B maps
        g.gemm_bf16_f32out(M, N, K, 1.0, A_d.data_ptr() + 2 * off, K, B_d.data_ptr() + 2 * off, N, 0.0,
                           C.data_ptr(), N, s)
        if i % 233 == 0 or i == 699:
            torch.cuda.synchronize()
            Ai = A_all[off:off + M * K].view(M, K)
            Bi = B_all[off:off + K * N].view(K, N)
            ref = oracle.gemm(Ai, Bi, 1.0, 0.0, None)
            err = oracle.normwise_error(C.cpu(), ref, oracle.abs_product_max(Ai, Bi))
            assert err <= oracle.TOL_BF16_F32OUT, (i, err)
    status, where = g.device_status()
    assert status == 0, (status, where)
