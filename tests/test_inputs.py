"""The seeded input generators: determinism, shapes, and bf16 rounding."""
import math

import numpy as np

import torch

from roofline_driven_optimisation_gb300 import inputs


def test_same_seed_same_bytes():
    a = inputs.make("fp32_256")
    b = inputs.make("fp32_256")
    assert torch.equal(a.A, b.A) and torch.equal(a.B, b.B)
    assert a.C0 is None


def test_shapes_and_dtypes():
    c = inputs.make("decode_m4_down", K=512, N=96)
    assert c.A.shape == (4, 512) and c.B.shape == (512, 96) and c.C0.shape == (4, 96)
    assert c.A.dtype == torch.bfloat16 and c.C0.dtype == torch.bfloat16
    assert c.spec.beta == 1.0
    f = inputs.make("fp32_4096", M=64, N=32, K=16)
    assert f.A.dtype == torch.float32 and f.C0.shape == (64, 32)
    assert (f.spec.alpha, f.spec.beta) == (1.5, 0.5)


def test_uniform_range():
    c = inputs.make("fp32_256")
    assert float(c.A.min()) >= -1.0 and float(c.A.max()) < 1.0


def test_bf16_round_to_nearest_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even -> 1
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    # 1 + 2^-8 + 2^-20 is above the halfway point -> 1 + 2^-7
    x = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)],
                     dtype=torch.float32)
    y = inputs.round_to(x, "bf16").to(torch.float64).tolist()
    assert y == [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0]


def test_normal_scale():
    c = inputs.make("bf16_4096", M=256, N=256, K=4096)
    std = float(c.A.float().std())
    assert abs(std - 1 / math.sqrt(4096)) < 0.1 / math.sqrt(4096)
    d = inputs.make("prefill_o", M=64, N=512, K=512)
    assert abs(float(d.B.float().std()) - 0.02) < 0.002
    assert abs(float(d.A.float().std()) - 1.0) < 0.05


def test_workload_table():
    assert inputs.spec("prefill_lm").N == 32000
    assert inputs.spec("decode_m16_down").K == 11008
    assert {inputs.spec(f"decode_m{m}_qkv").M for m in (1, 4, 16)} == {1, 4, 16}


def test_fp8_operands_are_seeded_codes():
    from oracle import fp8
    c1 = inputs.make_fp8(33, 40, 64, inputs.FP8_E4M3, inputs.FP8_E5M2, seed=3, beta=0.5)
    c2 = inputs.make_fp8(33, 40, 64, inputs.FP8_E4M3, inputs.FP8_E5M2, seed=3, beta=0.5)
    assert c1.A.dtype == torch.uint8 and c1.B.dtype == torch.uint8
    assert torch.equal(c1.A, c2.A) and torch.equal(c1.B, c2.B) and torch.equal(c1.C0, c2.C0)
    a = fp8.decode(c1.A, fp8.E4M3)
    b = fp8.decode(c1.B, fp8.E5M2)
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b))
    assert 0.5 < a.std() < 1.5 and 0.5 < b.std() < 1.5
    assert c1.alpha == 1 / 8


def test_int4_weights_pack_and_spread():
    from oracle import int4
    c = inputs.make_int4(256, 64, group=128, zero=8, seed=1)
    assert c.q.shape == (256, 32) and c.q.dtype == torch.uint8
    assert c.scales.shape == (2, 64) and c.scales.dtype == torch.bfloat16
    codes = int4.unpack(c.q, 64)
    assert codes.min() == 0 and codes.max() == 15
    w = int4.dequant_exact(c.q, c.scales, 64, 128, 8)
    assert 0.012 < w.std() < 0.03
    assert torch.equal(inputs.make_int4(256, 64, seed=1).q, c.q)
