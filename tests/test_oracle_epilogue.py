"""Pins of the fp64 epilogue activations: identities and textbook values."""
import math

import numpy as np

import oracle
from oracle import epilogue as E


def test_values_at_known_points():
    # sigmoid(1) = 1/(1+e^-1); Phi(1) = 0.8413447460685429 (standard normal CDF)
    assert abs(E.activate(1.0, E.SILU) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(E.activate(1.0, E.GELU) - 0.8413447460685429) < 1e-15
    assert E.activate(0.0, E.SILU) == 0.0 and E.activate(0.0, E.GELU) == 0.0
    assert list(E.activate([-2.0, 0.0, 3.5], E.RELU)) == [0.0, 0.0, 3.5]


def test_odd_part_identity():
    # silu(z) - silu(-z) = z and gelu(z) - gelu(-z) = z (sigmoid and Phi are
    # complementary about 0): a dropped factor or sign fails this
    z = np.linspace(-12, 12, 97)
    for act in (E.SILU, E.GELU):
        d = E.activate(z, act) - E.activate(-z, act)
        assert np.max(np.abs(d - z)) < 1e-12


def test_limits():
    assert abs(E.activate(40.0, E.SILU) - 40.0) < 1e-12
    assert abs(E.activate(-40.0, E.SILU)) < 1e-12
    assert abs(E.activate(10.0, E.GELU) - 10.0) < 1e-12
    assert abs(E.activate(-10.0, E.GELU)) < 1e-12
    assert E.activate(-1000.0, E.SILU) == 0.0   # no overflow to NaN


def test_gemm_epilogue_composition():
    rng = np.random.default_rng(3)
    A = rng.integers(-4, 5, size=(5, 7)).astype(np.float64)
    B = rng.integers(-4, 5, size=(7, 6)).astype(np.float64)
    C0 = rng.integers(-4, 5, size=(5, 6)).astype(np.float64)
    bias = np.arange(6, dtype=np.float64) - 2.5
    z = 1.5 * (A @ B) + 0.5 * C0 + bias   # integer/dyadic: exact
    got = E.gemm_epilogue(A, B, 1.5, 0.5, C0, bias, E.RELU)
    assert np.array_equal(got, np.maximum(z, 0.0))
    assert np.array_equal(E.gemm_epilogue(A, B, 1.5, 0.5, C0, bias, E.NONE), z)


def test_swiglu_reduces_to_products():
    rng = np.random.default_rng(4)
    A = rng.standard_normal((4, 9))
    Bg = rng.standard_normal((9, 5))
    Bu = rng.standard_normal((9, 5))
    g = oracle.gemm(A, Bg)
    u = oracle.gemm(A, Bu)
    got = E.swiglu(A, Bg, Bu)
    assert np.allclose(got, g / (1 + np.exp(-g)) * u, rtol=1e-15, atol=0)
    # a zero up-projection gives zero; an identity-like gate at large g gives g*u
    assert np.array_equal(E.swiglu(A, Bg, np.zeros_like(Bu)), np.zeros((4, 5)))
