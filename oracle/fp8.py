"""8-bit floating-point GEMM oracle: TEST INFRASTRUCTURE ONLY (see
``oracle/__init__``).

The contraction is the pages' C = sum_k A[:,k] B[k,:] (OCANNL "Module
Ir.Schedule", Tensorize; LuisaCompute "Pipelines and stage boundaries", the
k-tile example) on operands stored as 8-bit floating-point codes.  TVM
"Tensor Layout" (Scale factors, SFA / SFB) names 8-bit floating point as the
element type of its block-scaled GEMM but does not define the encodings; the
definitions followed here are the two formats of the OCP 8-bit floating point
specification (OFP8):

* E4M3: sign bit 7, exponent bits 6-3 with bias 7, mantissa bits 2-0.
  Exponent field 0 is subnormal, (-1)^s 2^-6 (m/8); otherwise normal,
  (-1)^s 2^(e-7) (1 + m/8); the code with every exponent and mantissa bit set
  (S.1111.111) is NaN, and there is no infinity (largest finite 448).
* E5M2: sign bit 7, exponent bits 6-2 with bias 15, mantissa bits 1-0.
  Exponent field 0 is subnormal, (-1)^s 2^-14 (m/4); exponent field 31 is
  infinity (m = 0) or NaN (m != 0); otherwise (-1)^s 2^(e-15) (1 + m/4).

Every finite code is an exact fp64 value.  A product of two E4M3 values has
8 significant bits between 2^-18 and 2^18, so a sum of K of them needs at
most 44 + log2(K) bits and the fp64 matmul below is exact for K < 2^9; with
E5M2's wider exponent range a sum can need more than fp64's 53 bits, and the
oracle is then within fp64 rounding (2^-53 relative per operation), far
below the GEMM's tolerance.

Pinned by ``tests/test_fp8_oracle.py``: all 256 codes of both formats against
an independent decoder (PyTorch's float8 dtypes), the specification's named
values (largest finite, smallest normal and subnormal, signed zero, NaN and
infinity codes), brute force with exact fractions on tiny products, and
planted mistakes (a wrong exponent bias, swapped formats) that the pins catch.
"""
from __future__ import annotations

import math

import numpy as np

from .epilogue import apply_epilogue_f64

E4M3 = 0
E5M2 = 1


def decode_e4m3(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


def decode_e5m2(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 2) & 0x1F
    m = code & 0x3
    if e == 0x1F:
        return s * math.inf if m == 0 else math.nan
    if e == 0:
        return s * math.ldexp(m / 4.0, -14)
    return s * math.ldexp(1.0 + m / 4.0, e - 15)


def table(fmt: int) -> np.ndarray:
    """fp64 value of each of the 256 codes of a format."""
    dec = decode_e4m3 if fmt == E4M3 else decode_e5m2
    return np.array([dec(c) for c in range(256)], dtype=np.float64)


def decode(codes, fmt: int) -> np.ndarray:
    """uint8 codes (any shape) -> fp64 values."""
    return table(fmt)[np.asarray(codes, dtype=np.uint8)]


def gemm_fp8_f64(A_codes, Bt_codes, fmt_a: int, fmt_b: int) -> np.ndarray:
    """C = A @ B in fp64 for A [.., M, K] and B given transposed, Bt [.., N, K]
    (the K-major layout of the library's 8-bit path)."""
    A = decode(A_codes, fmt_a)
    Bt = decode(Bt_codes, fmt_b)
    return np.matmul(A, np.swapaxes(Bt, -1, -2))


def gemm_fp8_epilogue_f64(A_codes, Bt_codes, fmt_a: int, fmt_b: int, **ep) -> np.ndarray:
    """The 8-bit GEMM followed by the fused epilogue of ``oracle.epilogue``."""
    return apply_epilogue_f64(gemm_fp8_f64(A_codes, Bt_codes, fmt_a, fmt_b), **ep)
