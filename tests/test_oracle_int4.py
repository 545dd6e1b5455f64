"""Pins of the INT4 weight decoding: the nibble order of the pages' example,
hand-computed values, zero points, groups, and the single bf16 rounding."""
import numpy as np
import torch

from oracle import int4


def test_nibble_order_low_first():
    # byte 0xA3 holds 3 (first element, low nibble) then 10 (high nibble)
    q = np.array([[0xA3, 0x0F]], dtype=np.uint8)
    assert int4.unpack(q, 4).tolist() == [[3, 10, 15, 0]]
    assert int4.unpack(q, 3).tolist() == [[3, 10, 15]]


def test_hand_values_with_groups_and_zero_point():
    q = np.array([[0x21], [0x43], [0xF0]], dtype=np.uint8)      # rows k=0,1,2; 2 columns
    s = torch.tensor([[0.5, 2.0], [0.25, -1.0]], dtype=torch.bfloat16)   # G = 2
    w = int4.dequant_exact(q, s, 2, group=2, zero=8)
    # k=0: codes (1, 2); k=1: (3, 4) -> group 0; k=2: (0, 15) -> group 1
    assert w.tolist() == [[0.5 * -7, 2.0 * -6], [0.5 * -5, 2.0 * -4], [0.25 * -8, -1.0 * 7]]
    # zero point 0 is the pages' plain scale * code
    assert int4.dequant_exact(q, s, 2, 2, 0)[2].tolist() == [0.0, -15.0]


def test_bf16_rounding_is_single_and_nearest_even():
    # scale 1 + 2^-7 (exact in bf16) times 15 = 15 + 15/128 needs 11 bits;
    # bf16 keeps 8: 15.1171875 -> nearest bf16 is 15.125
    s = torch.tensor([[1.0 + 2.0 ** -7]], dtype=torch.bfloat16)
    q = np.array([[0x0F]], dtype=np.uint8)
    assert int4.dequant_exact(q, s, 1, 1, 0)[0, 0] == 15.1171875
    assert int4.dequant_bf16(q, s, 1, 1, 0)[0, 0].item() == 15.125
    # every code times every power-of-two scale is exact
    codes = np.arange(16, dtype=np.uint8).reshape(1, 16)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s2 = torch.full((1, 16), 0.125, dtype=torch.bfloat16)
    assert int4.dequant_bf16(packed, s2, 16, 1, 8).float().tolist() == [[(c - 8) / 8 for c in range(16)]]


def test_gemm_w4_is_gemm_of_the_dequantised_weight():
    rng = np.random.default_rng(2)
    A = rng.integers(-3, 4, size=(3, 4)).astype(np.float64)
    q = rng.integers(0, 256, size=(4, 3)).astype(np.uint8)
    s = torch.tensor([[1.0, 0.5, 2.0, 4.0, 1.0, 0.25]] * 2, dtype=torch.bfloat16)
    got = int4.gemm_w4(A, q, s, 6, group=2, zero=8)
    W = int4.dequant_exact(q, s, 6, 2, 8)   # powers of two: the bf16 rounding is exact
    assert np.array_equal(got, A @ W)


def test_kmajor_repack_slot_order():
    # column 0 holds k = 0..7 -> codes 1..8; column 1 holds 15 everywhere
    K, N = 8, 2
    codes = np.stack([np.arange(1, 9), np.full(8, 15)], axis=1)
    q = (codes[:, 0] | (codes[:, 1] << 4)).astype(np.uint8).reshape(K, 1)
    r = int4.repack_kmajor(q, K, N)
    assert r.shape == (2, 4)
    w0 = int.from_bytes(r[0].tobytes(), "little")
    # slots 0..7 hold k = 0,2,4,6,1,3,5,7 -> codes 1,3,5,7,2,4,6,8
    assert [(w0 >> (4 * s)) & 0xF for s in range(8)] == [1, 3, 5, 7, 2, 4, 6, 8]
    # bits 0-3 and 16-19 of (word >> 4i) are k = 2i and 2i + 1
    for i in range(4):
        assert ((w0 >> (4 * i)) & 0xF, (w0 >> (4 * i + 16)) & 0xF) == (2 * i + 1, 2 * i + 2)
    assert int.from_bytes(r[1].tobytes(), "little") == 0xFFFFFFFF


def test_kmajor_repack_round_trip_and_padding():
    rng = np.random.default_rng(9)
    K, N = 21, 6
    codes = rng.integers(0, 16, size=(K, N))
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    r = int4.repack_kmajor(q, K, N)
    assert r.shape == (N, 12)
    words = r.view("<u4").reshape(N, 3)
    back = np.zeros((24, N), dtype=np.int64)
    for s, dk in enumerate(int4.SLOT_K):
        back[dk::8] = ((words >> (4 * s)) & 0xF).T
    assert np.array_equal(back[:K], codes) and not back[K:].any()


def test_exact_w4_gemm_differs_from_rounded_only_by_the_rounding():
    rng = np.random.default_rng(4)
    A = rng.standard_normal((3, 64))
    q = rng.integers(0, 256, size=(64, 4)).astype(np.uint8)
    s = torch.tensor(rng.uniform(0.003, 0.006, size=(1, 8)), dtype=torch.bfloat16)
    exact = int4.gemm_w4_exact(A, q, s, 8, 64, 8)
    W = int4.dequant_exact(q, s, 8, 64, 8)
    assert np.allclose(exact, A @ W, rtol=1e-13, atol=1e-15)
    rounded = int4.gemm_w4(A, q, s, 8, 64, 8)
    scale = np.abs(A) @ np.abs(W)
    assert np.max(np.abs(rounded - exact) / scale.max()) <= 2.0 ** -9


def test_tiled_layout_places_each_tile_contiguously():
    rng = np.random.default_rng(12)
    K, N = 130, 200                       # 3 K tiles (last partial), 2 column tiles
    codes = rng.integers(0, 16, size=(K, N))
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    t = int4.repack_tiled(q, K, N)
    assert t.size == int4.tiled_bytes(K, N) == 2 * 3 * 4096
    rows = int4.repack_kmajor(q, K, N)    # N x 68
    for n in (0, 127, 128, 199):
        for kt in range(3):
            blk = ((n // 128) * 3 + kt) * 4096 + (n % 128) * 32
            want = np.zeros(32, dtype=np.uint8)
            seg = rows[n, kt * 32:(kt + 1) * 32]
            want[: seg.size] = seg
            assert np.array_equal(t[blk:blk + 32], want)
    # the padding columns of the last tile are zero
    assert not t[(1 * 3 + 0) * 4096 + 72 * 32:(1 * 3 + 1) * 4096].any()
