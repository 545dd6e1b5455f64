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


def test_swiglu_worked_values():
    # K = 1: g = 2, u = 3 gives silu(2) * 3 with sigmoid(2) = 0.8807970779778823;
    # the gate, not the up projection, goes through silu (swapped: 5.7154...)
    A = np.array([[2.0]])
    got = E.swiglu(A, np.array([[1.0]]), np.array([[1.5]]))
    assert abs(got[0, 0] - 2.0 * 0.8807970779778823 * 3.0) < 1e-14
    # a very negative gate switches the output off whatever the up projection
    assert abs(E.swiglu(A, np.array([[-30.0]]), np.array([[100.0]]))[0, 0]) < 1e-20


def test_silu_slope_bound():
    z = np.linspace(-20, 20, 400001)
    s = 1.0 / (1.0 + np.exp(-z))
    slope = s * (1.0 + z * (1.0 - s))
    assert slope.max() <= E.SILU_SLOPE_BOUND
    assert slope.max() > 1.09            # the bound is tight, not a loose guess
    assert abs(z[slope.argmax()] - 2.40) < 0.01


def test_swiglu_error_scale_closed_form():
    # g = 1 - 1 = 0 with sum|A||Bg| = 2; u = 2 + 3 = 5 with sum|A||Bu| = 5:
    # scale = 1.1 * 5 * 2 + silu(0) * 5 = 11 -- the gate term alone carries it
    A = np.array([[1.0, 1.0]])
    s = E.swiglu_error_scale(A, np.array([[1.0], [-1.0]]), np.array([[2.0], [3.0]]))
    assert abs(s - 11.0) < 1e-12
    # u = 0 exactly: only the up term remains, silu(2) * sum|A||Bu| = silu(2) * 2
    s = E.swiglu_error_scale(A, np.array([[1.0], [1.0]]), np.array([[1.0], [-1.0]]))
    assert abs(s - 2.0 * 0.8807970779778823 * 2.0) < 1e-12


def test_swiglu_error_scale_bounds_perturbations():
    # perturbing g and u by at most eps * sum|A||B| elementwise moves the
    # output by at most eps * scale (first order), and |output| <= scale
    rng = np.random.default_rng(11)
    A = rng.standard_normal((6, 40))
    Bg = rng.standard_normal((40, 7)) * 0.3
    Bu = rng.standard_normal((40, 7)) * 0.3
    scale = E.swiglu_error_scale(A, Bg, Bu)
    g, u = A @ Bg, A @ Bu
    Sg, Su = np.abs(A) @ np.abs(Bg), np.abs(A) @ np.abs(Bu)
    out = E.activate(g, E.SILU) * u
    assert np.abs(out).max() <= scale
    eps = 1e-7
    for _ in range(20):
        dg = rng.uniform(-1, 1, g.shape) * eps * Sg
        du = rng.uniform(-1, 1, u.shape) * eps * Su
        moved = E.activate(g + dg, E.SILU) * (u + du) - out
        assert np.abs(moved).max() <= eps * scale * (1 + 1e-6)
