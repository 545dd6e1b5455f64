"""gemm_f32_noalloc against gemm_f32 through the C ABI.

gemm_f32_noalloc runs the plan and kernels of gemm_f32 with the stream-K
tail's scratch in a static device array.  Each case runs gemm_f32 once, then
gemm_f32_noalloc twice in a row on the same stream (the second call reuses
the scratch the first one left), and holds both results to the FP32
tolerance of the parity tests against gemm_f32's -- and, as the header
states, to the same bits.  The file is named to be collected last, and each
case also passes alone in a fresh process (the first call on the device sets
up the scratch's address)."""
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _args(A, B, C, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    return (M, N, K, float(alpha), A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
            float(beta), C.data_ptr(), C.stride(0))


def _normwise(C, C_ref, A, B, C0, alpha, beta):
    # the parity tests' error scale: max(|alpha| sum_k |A||B| + |beta||C0|),
    # here in fp64 on the device (both results come from the GPU)
    scale = (abs(alpha) * (A.double().abs() @ B.double().abs()) + abs(beta) * C0.double().abs()).max()
    return ((C.double() - C_ref.double()).abs().max() / scale).item()


# (M, N, K, forced tile width, expect a stream-K tail)
CASES = [
    (300, 520, 1024, 256, True),      # 9 wide tiles, all in the tail (36 CTAs)
    (2048, 2048, 4096, 0, True),      # 128 wide tiles: the tail on every SM
    (4096, 4096, 4096, 0, True),      # 3 whole waves + a 56-tile tail
    (2560, 2048, 1024, 128, False),   # narrow tiles, cluster split: no scratch
    (1000, 1004, 1001, 0, False),     # lda = 1001, not a multiple of 4: generic kernel
]


@pytest.mark.parametrize("M,N,K,tile_n,stream_k", CASES)
def test_noalloc_matches_gemm_f32(cuda_lib, M, N, K, tile_n, stream_k):
    g = cuda_lib
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, device=dev, generator=gen)
    B = torch.randn(K, N, device=dev, generator=gen)
    C0 = torch.randn(M, N, device=dev, generator=gen)
    alpha, beta = 1.5, 0.5
    C_ref, C1, C2 = C0.clone(), C0.clone(), C0.clone()
    s = torch.cuda.current_stream().cuda_stream
    g.force_tile_n(tile_n)
    try:
        g.gemm_f32(*_args(A, B, C_ref, alpha, beta), s)
        ref_split = g.last_k_split()
        torch.cuda.synchronize()
        g.gemm_f32_noalloc(*_args(A, B, C1, alpha, beta), s)
        path, tile, split = g.last_path(), g.last_tile_n(), g.last_k_split()
        free_before, _ = torch.cuda.mem_get_info()
        g.gemm_f32_noalloc(*_args(A, B, C2, alpha, beta), s)
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
    finally:
        g.force_tile_n(0)
    status, where = g.device_status()
    assert status == 0, f"device status {status} at site {where}"
    if stream_k:
        assert path == g.PATH_F32_SIMT and tile == 256 and split > 1
        assert split == ref_split
    assert free_after == free_before, "gemm_f32_noalloc changed the device's free memory"
    for C in (C1, C2):
        err = _normwise(C, C_ref, A, B, C0, alpha, beta)
        assert err <= oracle.TOL_F32, f"normwise difference {err:.3e} > {oracle.TOL_F32:g}"
        assert torch.equal(C, C_ref)


def test_noalloc_rejects_bad_arguments(cuda_lib):
    g = cuda_lib
    A = torch.zeros(4, 4, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32_noalloc(-1, 4, 4, 1.0, A.data_ptr(), 4, A.data_ptr(), 4, 0.0, A.data_ptr(), 4, s)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f32_noalloc(4, 4, 4, 1.0, A.data_ptr(), 2, A.data_ptr(), 4, 0.0, A.data_ptr(), 4, s)
    assert e.value.code == g.GEMM_ERR_INVALID_ARG
