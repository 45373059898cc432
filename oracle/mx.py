"""Block-scaled 8-bit GEMM oracle: TEST INFRASTRUCTURE ONLY (see
``oracle/__init__``).

TVM "Tensor Layout" (Scale factors, SFA / SFB) describes the block-scaled
GEMM: each operand carries one scale factor per block of 32 consecutive
elements along K, kept in tensor memory next to the accumulator.  The pages
do not define the encodings; the definitions followed here are those of the
OCP Microscaling (MX) specification for MXFP8: elements are OFP8 E4M3 or
E5M2 codes (``oracle.fp8``), and a scale factor is an E8M0 code e, the value
2^(e - 127) (e = 255 is NaN).  The product is

    C[m][n] = sum_k (A[m][k] * SA[m][k // 32]) * (B[k][n] * SB[n][k // 32])

with B given transposed (Bt[n][k]), SA [M, ceil(K/32)] and SB [N, ceil(K/32)],
evaluated in fp64: every scaled element is an exact fp64 value, so the only
rounding is the fp64 summation (exact while the partial sums fit in 53 bits).

Pinned by ``tests/test_mx_oracle.py``: the E8M0 decoder against PyTorch's
float8_e8m0fnu for all 256 codes, brute force with exact fractions,
unit scales reducing to ``oracle.fp8``, and per-block scaling laws.
"""
from __future__ import annotations

import math

import numpy as np

from . import fp8

BLOCK = 32  # elements of K per scale factor


def decode_e8m0(code: int) -> float:
    return math.nan if code == 0xFF else math.ldexp(1.0, code - 127)


def e8m0_table() -> np.ndarray:
    return np.array([decode_e8m0(c) for c in range(256)], dtype=np.float64)


def scaled(codes, fmt: int, sf) -> np.ndarray:
    """fp64 values of [.., R, K] codes times their rows' block scales
    sf [.., R, ceil(K/32)] (E8M0 codes)."""
    v = fp8.decode(codes, fmt)
    s = e8m0_table()[np.asarray(sf, dtype=np.uint8)]
    K = v.shape[-1]
    s_full = np.repeat(s, BLOCK, axis=-1)[..., :K]
    return v * s_full


def gemm_mx_f64(A_codes, Bt_codes, fmt_a: int, fmt_b: int, sfa, sfb) -> np.ndarray:
    """C = (A scaled by SA) @ (B scaled by SB), B given transposed."""
    A = scaled(A_codes, fmt_a, sfa)
    Bt = scaled(Bt_codes, fmt_b, sfb)
    return np.matmul(A, np.swapaxes(Bt, -1, -2))
