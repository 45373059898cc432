"""Pins of the fused-epilogue oracle (CPU only)."""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import epilogue as ep

scipy_special = pytest.importorskip("scipy.special")


def test_identity_epilogue_returns_c():
    C = np.random.default_rng(0).standard_normal((5, 7))
    assert np.array_equal(ep.apply_epilogue_f64(C), C)


def test_relu_closed_form():
    x = np.array([-3.0, -0.0, 0.0, 1e-300, 2.5])
    assert np.array_equal(ep.activation_f64(x, ep.ACT_RELU), np.array([0.0, 0.0, 0.0, 1e-300, 2.5]))


@pytest.mark.parametrize("act", [ep.ACT_GELU_TANH, ep.ACT_SILU])
def test_odd_part_identity(act):
    """Both x*s(x) activations with s(x) + s(-x) = 1 satisfy
    act(x) - act(-x) = x exactly in real arithmetic."""
    x = np.linspace(-12, 12, 2001)
    d = ep.activation_f64(x, act) - ep.activation_f64(-x, act)
    assert np.allclose(d, x, rtol=0, atol=1e-12)


@pytest.mark.parametrize("act", [ep.ACT_GELU_TANH, ep.ACT_SILU])
def test_limits_and_zero(act):
    big = np.array([40.0, 100.0])
    assert np.allclose(ep.activation_f64(big, act), big, rtol=1e-12)
    assert np.allclose(ep.activation_f64(-big, act), 0.0, atol=1e-12)
    assert ep.activation_f64(np.array([0.0]), act)[0] == 0.0


def test_gelu_tanh_close_to_erf_gelu():
    """The tanh form stays within 5e-4 of x * Phi(x) (a library routine)."""
    x = np.linspace(-8, 8, 4001)
    exact = 0.5 * x * (1.0 + scipy_special.erf(x / math.sqrt(2.0)))
    assert np.max(np.abs(ep.activation_f64(x, ep.ACT_GELU_TANH) - exact)) < 5e-4


def test_silu_is_x_times_logistic():
    x = np.linspace(-30, 30, 3001)
    assert np.allclose(ep.activation_f64(x, ep.ACT_SILU), x * scipy_special.expit(x), rtol=1e-14, atol=1e-300)


def test_epilogue_order_bias_act_residual():
    """bias goes in before the activation, the residual after it."""
    C = np.array([[-1.0, 2.0]])
    bias = np.array([3.0, -5.0])
    R = np.array([[10.0, 20.0]])
    D = ep.apply_epilogue_f64(C, alpha=2.0, bias=bias, act=ep.ACT_RELU, beta=0.5, residual=R)
    # relu(2*-1 + 3) + 5 = 6 ; relu(2*2 - 5) + 10 = 10
    assert np.array_equal(D, np.array([[6.0, 10.0]]))


def test_batched_bias():
    C = np.zeros((2, 3, 4))
    bias = np.arange(8.0).reshape(2, 4)
    D = ep.apply_epilogue_f64(C, bias=bias)
    assert np.array_equal(D[1, 2], bias[1]) and np.array_equal(D[0, 1], bias[0])
