"""INT4 weight-only decode GEMM and the tiled repack, through the C ABI.
The repack is compared bit for bit with the oracle's; the GEMM with the fp64
GEMM on the exact weight s * (q - z): its products are exact (bf16 X times the
integers q - z), so the tolerances are those of the bf16-input GEMM with the
scale max(|alpha| sum|X||W| + |beta||C0|)."""
import numpy as np
import pytest
import torch

import oracle
import roofline_driven_optimisation_gb300 as g
from oracle import int4
from roofline_driven_optimisation_gb300 import inputs

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32
TOL = {BF16: oracle.TOL_BF16_OUT, F32: oracle.TOL_BF16_F32OUT}


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _expected_split(N, K, group):
    tiles = -(-N // 128)
    groups = -(-K // group)
    s = 1
    while s * 2 <= 8 and tiles * s * 2 <= 2 * _sms():
        s *= 2
    while s > 1 and s > groups:
        s //= 2
    return s


@pytest.mark.parametrize("K,N", [(64, 128), (21, 7), (4096, 256), (100, 33), (130, 200)])
def test_repack_bit_exact(cuda_lib, K, N):
    c = inputs.make_int4(K, N + (N % 2), group=32, zero=8, seed=K + N)
    q = c.q[:, : (N + 1) // 2].contiguous()
    size = g.gemm_w4_packed_bytes(K, N)
    assert size == int4.tiled_bytes(K, N)
    buf = torch.full((size + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    g.gemm_int4_repack(q.cuda().data_ptr(), K, N, q.shape[1], buf.data_ptr(),
                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    assert np.array_equal(got[:size], int4.repack_tiled(q, K, N))
    assert (got[size:] == 0xAB).all()        # nothing past the layout is written


def _case(M, N, K, group=128, zero=8, seed=11, beta=1.0):
    w = inputs.make_int4(K, N, group=group, zero=zero, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    X = torch.randn((M, K), generator=gen).to(BF16)
    C0 = torch.randn((M, N), generator=gen).to(BF16) if beta != 0 else None
    return w, X, C0


def _run(w, X, C0, out, alpha=1.0, beta=1.0, x_off=0):
    M, K = X.shape
    N = w.N
    qk = g.int4_repack(w.q.cuda(), K, N)
    flat = torch.zeros(x_off + M * K + 8, dtype=BF16)
    flat[x_off:x_off + M * K] = X.reshape(-1)
    Xd = flat.cuda()
    C = C0.to(out).cuda() if C0 is not None else torch.full((M, N), float("nan"), dtype=out, device="cuda")
    fn = g.gemm_w4a16 if out == BF16 else g.gemm_w4a16_f32out
    fn(M, N, K, alpha, Xd.data_ptr() + 2 * x_off, K, qk.data_ptr(), w.scales.cuda().data_ptr(),
       w.scales.shape[1], w.group, w.zero, beta, C.data_ptr(), N, torch.cuda.current_stream().cuda_stream)
    ran, split = g.last_path(), g.last_k_split()
    torch.cuda.synchronize()
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"
    return C.cpu(), ran, split


def _check(w, X, C0, out, alpha=1.0, beta=1.0, **kw):
    C, ran, split = _run(w, X, C0, out, alpha, beta, **kw)
    C0e = C0.to(out) if C0 is not None else None
    ref = int4.gemm_w4_exact(X, w.q, w.scales, w.N, w.group, w.zero, alpha, beta, C0e)
    W = int4.dequant_exact(w.q, w.scales, w.N, w.group, w.zero)
    den = oracle.normwise_denominator(X, W, alpha, beta, C0e)
    err = oracle.normwise_error(C, ref, den if den else 1.0)
    assert err <= TOL[out], f"normwise error {err:.3e} > {TOL[out]:g} (path {g.PATH_NAMES.get(ran)})"
    return err, ran, split


@pytest.mark.parametrize("out", [BF16, F32])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_llama_gate_shape(cuda_lib, out, M):
    # LLaMA-7B gate/up weight (K 4096, N 11008), group 128, zero point 8, beta 1
    w, X, C0 = _case(M, 11008, 4096)
    _, ran, split = _check(w, X, C0, out)
    assert ran == g.PATH_W4 and split == _expected_split(11008, 4096, 128)


@pytest.mark.parametrize("M,N,K,group", [(3, 256, 4096, 128), (16, 200, 4000, 128), (5, 4096, 1024, 64),
                                         (2, 512, 2048, 256), (7, 384, 512, 4096), (1, 136, 64, 64)])
def test_splits_groups_and_tails(cuda_lib, M, N, K, group):
    # N = 256: two column tiles, split 8; K = 4000: a partial last stage and
    # group; group >= K: one group, no split; N = 136: a ragged second tile
    w, X, C0 = _case(M, N, K, group=group, seed=M + N)
    for out in (BF16, F32):
        _, ran, split = _check(w, X, C0, out)
        assert ran == g.PATH_W4 and split == _expected_split(N, K, group)


def test_alpha_beta_zero_point(cuda_lib):
    w, X, C0 = _case(6, 384, 1024, group=128, zero=0, seed=3)
    _check(w, X, C0, F32, alpha=0.5, beta=-2.0)
    w, X, _ = _case(6, 384, 1024, group=64, zero=15, seed=4, beta=0.0)
    _, ran, _ = _check(w, X, None, BF16, alpha=1.5, beta=0.0)
    assert ran == g.PATH_W4


@pytest.mark.parametrize("M,N,K,group,x_off", [(17, 256, 512, 128, 0), (4, 256, 512, 100, 0),
                                               (4, 256, 512, 128, 3), (2, 30, 24, 8, 0)])
def test_generic_kernel(cuda_lib, M, N, K, group, x_off):
    # M > 16, a group size that is not a multiple of 64, an unaligned X
    w, X, C0 = _case(M, N, K, group=group, seed=N + K)
    for out in (BF16, F32):
        _, ran, _ = _check(w, X, C0, out, x_off=x_off)
        assert ran == g.PATH_GENERIC


def test_forced_generic_agrees(cuda_lib):
    w, X, C0 = _case(8, 512, 1024, seed=5)
    fast, ran, _ = _run(w, X, C0, F32)
    assert ran == g.PATH_W4
    g.force_path(g.PATH_GENERIC)
    try:
        slow, ran, _ = _run(w, X, C0, F32)
    finally:
        g.force_path(g.PATH_AUTO)
    assert ran == g.PATH_GENERIC
    assert torch.allclose(fast, slow, rtol=0, atol=1e-4 * float(slow.abs().max()))


@pytest.mark.parametrize("M", [1, 16])
def test_llama_down_shape(cuda_lib, M):
    # K 11008: 86 groups of 128 over a split-K cluster, ranks with odd stage counts
    w, X, C0 = _case(M, 512, 11008, seed=M + 7)
    _, ran, split = _check(w, X, C0, BF16)
    assert ran == g.PATH_W4 and split > 1


def test_back_to_back_calls_match_synchronised_calls(cuda_lib):
    # the LLaMA-7B weight shapes (fewer columns) at M = 1, 4, 16, launched back
    # to back on one stream as a decode step does: every result must equal the
    # same call made alone
    st = torch.cuda.current_stream().cuda_stream
    calls = []
    for m in (1, 4, 16):
        for K, N in ((4096, 1536), (4096, 512), (4096, 1376), (11008, 512), (4096, 4000)):
            w, X, C0 = _case(m, N, K, seed=m * 31 + N + K)
            qk = g.int4_repack(w.q.cuda(), K, N)
            calls.append((m, N, K, X.cuda(), qk, w.scales.cuda(), C0.cuda()))

    def run(sync):
        outs = []
        for m, N, K, X, qk, sc, C0 in calls:
            C = C0.clone()
            g.gemm_w4a16(m, N, K, 1.0, X.data_ptr(), K, qk.data_ptr(), sc.data_ptr(), N, 128, 8, 1.0,
                         C.data_ptr(), N, st)
            outs.append(C)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return [c.cpu() for c in outs]

    ref = run(True)
    for _ in range(3):
        got = run(False)
        status, where = g.device_status()
        assert status == 0, (status, where)
        for a, b in zip(got, ref):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_deterministic(cuda_lib):
    w, X, C0 = _case(16, 1024, 4096, seed=6)
    a1, _, split = _run(w, X, C0, F32)
    a2, _, _ = _run(w, X, C0, F32)
    assert split > 1 and torch.equal(a1, a2)


def test_arguments(cuda_lib):
    st = torch.cuda.current_stream().cuda_stream
    X = torch.zeros((2, 64), dtype=BF16, device="cuda")
    qk = torch.zeros((4096,), dtype=torch.uint8, device="cuda")
    s = torch.ones((1, 128), dtype=BF16, device="cuda")
    C = torch.zeros((2, 128), dtype=BF16, device="cuda")
    base = [2, 128, 64, 1.0, X.data_ptr(), 64, qk.data_ptr(), s.data_ptr(), 128, 64, 8, 0.0,
            C.data_ptr(), 128, st]
    for idx, val, code in ((9, 0, g.GEMM_ERR_INVALID_ARG), (10, 16, g.GEMM_ERR_INVALID_ARG),
                           (5, 32, g.GEMM_ERR_INVALID_ARG), (7, s.data_ptr() + 1, g.GEMM_ERR_MISALIGNED),
                           (6, qk.data_ptr() + 4, g.GEMM_ERR_MISALIGNED)):
        args = list(base)
        args[idx] = val
        with pytest.raises(g.GemmError) as e:
            g.gemm_w4a16(*args)
        assert e.value.code == code
    # K = 0: C = beta * C
    C.fill_(2.0)
    args = list(base)
    args[2], args[11] = 0, 0.5
    g.gemm_w4a16(*args)
    torch.cuda.synchronize()
    assert torch.equal(C.float().cpu(), torch.ones((2, 128)))
