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

MXFP4 (the same block scaling on 4-bit elements): an element is an E2M1
code - sign bit 3, exponent bits 2-1 with bias 1, mantissa bit 0; exponent
field 0 is subnormal, (-1)^s (m/2); otherwise (-1)^s 2^(e-1) (1 + m/2); no
infinity or NaN, largest magnitude 6.  Two elements share a byte: element k
of a row is in byte k // 2, in the low nibble when k is even and in the high
nibble when k is odd (the library's storage convention for packed 4-bit
operands).  ``gemm_mxfp4_f64`` unpacks, decodes, scales and multiplies in
fp64 exactly as ``gemm_mx_f64`` does.

Pinned by ``tests/test_mx_oracle.py``: the E8M0 decoder against PyTorch's
float8_e8m0fnu for all 256 codes, brute force with exact fractions,
unit scales reducing to ``oracle.fp8``, and per-block scaling laws; the E2M1
decoder against the value list of the OCP MX specification and against the
OFP8 E4M3 decoder (every E2M1 value is an E4M3 value with the same sign,
exponent and mantissa), the nibble order, and brute force with exact
fractions.
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


def decode_e2m1(code: int) -> float:
    """fp64 value of a 4-bit E2M1 code (0..15)."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * (m / 2.0)
    return s * math.ldexp(1.0 + m / 2.0, e - 1)


def e2m1_table() -> np.ndarray:
    return np.array([decode_e2m1(c) for c in range(16)], dtype=np.float64)


def unpack_fp4(packed, K: int) -> np.ndarray:
    """[.., ceil(K/2)] bytes of packed E2M1 elements -> [.., K] codes (uint8):
    element 2i is the low nibble of byte i, element 2i + 1 the high nibble."""
    b = np.asarray(packed, dtype=np.uint8)
    lo = b & 0x0F
    hi = b >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(b.shape[:-1] + (2 * b.shape[-1],))
    return codes[..., :K]


def pack_fp4(codes) -> np.ndarray:
    """Inverse of ``unpack_fp4``: [.., K] codes (0..15) -> [.., ceil(K/2)]
    bytes (a missing odd element is packed as the code 0)."""
    c = np.asarray(codes, dtype=np.uint8)
    K = c.shape[-1]
    if K % 2:
        c = np.concatenate([c, np.zeros(c.shape[:-1] + (1,), np.uint8)], axis=-1)
    c = c.reshape(c.shape[:-1] + (-1, 2))
    return (c[..., 0] | (c[..., 1] << 4)).astype(np.uint8)


def scaled_fp4(packed, K: int, sf) -> np.ndarray:
    """fp64 values of packed E2M1 rows [.., R, ceil(K/2)] times their block
    scales sf [.., R, ceil(K/32)] (E8M0 codes)."""
    v = e2m1_table()[unpack_fp4(packed, K)]
    s = e8m0_table()[np.asarray(sf, dtype=np.uint8)]
    s_full = np.repeat(s, BLOCK, axis=-1)[..., :K]
    return v * s_full


def gemm_mxfp4_f64(A_packed, Bt_packed, K: int, sfa, sfb) -> np.ndarray:
    """C = (A scaled by SA) @ (B scaled by SB) for packed E2M1 A [.., M, K/2]
    and B given transposed, Bt [.., N, K/2]."""
    A = scaled_fp4(A_packed, K, sfa)
    Bt = scaled_fp4(Bt_packed, K, sfb)
    return np.matmul(A, np.swapaxes(Bt, -1, -2))
