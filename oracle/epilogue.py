"""Fused-epilogue oracle: TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

OCANNL "Module Ir.Schedule", Epilogue fusion: the elementwise tail that
follows a reduction - a bias add, an activation, a residual - is folded into
the accumulator's store-back; it never reorders the reduction.  The library
computes

    D[i][j] = act(alpha * C[i][j] + bias[j]) + beta * R[i][j]

where C = A B is the contraction.  This module evaluates that formula in
fp64 on the oracle's fp64 C, elementwise, in the order written.

Activations (fp64):
* relu(x)      = max(x, 0)
* gelu_tanh(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))
  (the tanh form of the Gaussian error linear unit)
* silu(x)      = x / (1 + exp(-x))

Pinned by ``tests/test_epilogue_oracle.py``: closed forms and limits, the
identity act(x) - act(-x) = x that both gelu_tanh and silu satisfy, erf-GELU
within its known tanh-approximation gap, scipy's logistic function, and the
identity epilogue.
"""
from __future__ import annotations

import math

import numpy as np

ACT_NONE = 0
ACT_RELU = 1
ACT_GELU_TANH = 2
ACT_SILU = 3
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu_tanh": ACT_GELU_TANH, "silu": ACT_SILU}

_GELU_K = math.sqrt(2.0 / math.pi)


def activation_f64(x: np.ndarray, act: int) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    if act == ACT_NONE:
        return x.copy()
    if act == ACT_RELU:
        return np.maximum(x, 0.0)
    if act == ACT_GELU_TANH:
        return 0.5 * x * (1.0 + np.tanh(_GELU_K * (x + 0.044715 * x * x * x)))
    if act == ACT_SILU:
        out = np.empty_like(x)
        pos = x >= 0
        out[pos] = x[pos] / (1.0 + np.exp(-x[pos]))
        ex = np.exp(x[~pos])  # x < 0: x * e^x / (1 + e^x), no overflow
        out[~pos] = x[~pos] * ex / (1.0 + ex)
        return out
    raise ValueError(f"unknown activation {act}")


def apply_epilogue_f64(C: np.ndarray, alpha: float = 1.0, bias=None, act: int = ACT_NONE,
                       beta: float = 0.0, residual=None) -> np.ndarray:
    """D = act(alpha*C + bias[None, :]) + beta*residual, all fp64.

    C: [..., M, N]; bias: [N] or [batch, N] (or None); residual: like C (or
    None, meaning no residual term)."""
    C = np.asarray(C, dtype=np.float64)
    x = alpha * C
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        x = x + (b[..., None, :] if b.ndim == C.ndim - 1 else b)
    y = activation_f64(x, act)
    if residual is not None:
        y = y + beta * np.asarray(residual, dtype=np.float64)
    return y
