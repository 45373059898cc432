"""Pins of the block-scaled 8-bit oracle (CPU only)."""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8, mx


def test_e8m0_every_code_matches_independent_decoder():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = mx.e8m0_table()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert mx.decode_e8m0(127) == 1.0 and mx.decode_e8m0(128) == 2.0 and mx.decode_e8m0(0) == 2.0 ** -127


def _frac_fp8(fmt, code):
    if fmt == fp8.E4M3:
        s, e, m, bias, mb = code >> 7, (code >> 3) & 15, code & 7, 7, 3
    else:
        s, e, m, bias, mb = code >> 7, (code >> 2) & 31, code & 3, 15, 2
    sign = -1 if s else 1
    if e == 0:
        return sign * Fraction(m, 1 << mb) * Fraction(2) ** (1 - bias)
    return sign * (1 + Fraction(m, 1 << mb)) * Fraction(2) ** (e - bias)


def _codes(fmt, rng, shape):
    t = fp8.table(fmt)
    return rng.choice(np.flatnonzero(np.isfinite(t)), size=shape).astype(np.uint8)


@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 0)])
def test_brute_force_fractions(fa, fb):
    rng = np.random.default_rng(11 + fa)
    M, N, K = 3, 2, 70  # three scale blocks, the last one ragged
    A, Bt = _codes(fa, rng, (M, K)), _codes(fb, rng, (N, K))
    sfa = rng.integers(120, 135, size=(M, 3)).astype(np.uint8)
    sfb = rng.integers(120, 135, size=(N, 3)).astype(np.uint8)
    got = mx.gemm_mx_f64(A, Bt, fa, fb, sfa, sfb)
    for i in range(M):
        for j in range(N):
            exact = sum(_frac_fp8(fa, int(A[i, k])) * Fraction(2) ** (int(sfa[i, k // 32]) - 127) *
                        _frac_fp8(fb, int(Bt[j, k])) * Fraction(2) ** (int(sfb[j, k // 32]) - 127)
                        for k in range(K))
            assert got[i, j] == float(exact), (i, j)


def test_unit_scales_reduce_to_the_unscaled_product():
    rng = np.random.default_rng(3)
    A, Bt = _codes(0, rng, (2, 9, 100)), _codes(0, rng, (2, 7, 100))
    one_a = np.full((2, 9, 4), 127, np.uint8)
    one_b = np.full((2, 7, 4), 127, np.uint8)
    assert np.array_equal(mx.gemm_mx_f64(A, Bt, 0, 0, one_a, one_b), fp8.gemm_fp8_f64(A, Bt, 0, 0))


def test_scaling_one_block_scales_its_contribution():
    """Raising the scale of A row i's block g by 1 doubles exactly that
    block's share of row i (a power of two is exact)."""
    rng = np.random.default_rng(5)
    M, N, K = 4, 5, 96
    A, Bt = _codes(0, rng, (M, K)), _codes(0, rng, (N, K))
    sfa = np.full((M, 3), 127, np.uint8)
    sfb = np.full((N, 3), 127, np.uint8)
    base = mx.gemm_mx_f64(A, Bt, 0, 0, sfa, sfb)
    block = fp8.decode(A, 0)[:, 32:64] @ fp8.decode(Bt, 0)[:, 32:64].T
    sfa2 = sfa.copy()
    sfa2[2, 1] = 128
    got = mx.gemm_mx_f64(A, Bt, 0, 0, sfa2, sfb)
    want = base.copy()
    want[2] += block[2]
    assert np.array_equal(got, want)


def test_planted_wrong_block_size_is_caught():
    rng = np.random.default_rng(9)
    A, Bt = _codes(0, rng, (3, 64)), _codes(0, rng, (2, 64))
    sfa = rng.integers(125, 130, size=(3, 2)).astype(np.uint8)
    sfb = rng.integers(125, 130, size=(2, 2)).astype(np.uint8)
    good = mx.gemm_mx_f64(A, Bt, 0, 0, sfa, sfb)
    old = mx.BLOCK
    try:
        mx.BLOCK = 16  # a planted mistake: blocks of 16 along K
        bad = mx.gemm_mx_f64(A, Bt, 0, 0, np.repeat(sfa, 2, axis=1), np.repeat(sfb, 2, axis=1))
        shifted = mx.gemm_mx_f64(A, Bt, 0, 0, np.concatenate([sfa, sfa], 1), np.concatenate([sfb, sfb], 1))
    finally:
        mx.BLOCK = old
    assert np.array_equal(bad, good)        # the same scales repeated per 16: same product
    assert not np.array_equal(shifted, good)  # but a 16-block reading of 32-block scales differs


# ------------------------------------------------------------ MXFP4 (E2M1)
# The E2M1 values as the OCP Microscaling specification lists them (codes
# 0..7; codes 8..15 are their negatives): 0, 0.5, 1, 1.5, 2, 3, 4, 6.
E2M1_SPEC = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_every_code_matches_the_specification_list():
    t = mx.e2m1_table()
    assert list(t[:8]) == E2M1_SPEC
    assert list(t[8:]) == [-v for v in E2M1_SPEC]
    assert np.signbit(t[8]) and not np.signbit(t[0])  # the two zeros


def test_e2m1_values_are_e4m3_values_with_the_same_fields():
    """An E2M1 code (s, e, m) has the value of the E4M3 code with the same
    sign, the exponent moved from bias 1 to bias 7, and the mantissa bit as
    E4M3's top mantissa bit (subnormal E2M1 0.5 = E4M3 2^-1)."""
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        if e == 0 and m == 0:
            ref = -0.0 if s else 0.0
        elif e == 0:
            ref = fp8.decode_e4m3((s << 7) | (6 << 3))  # 0.5 = 2^(6-7)
        else:
            ref = fp8.decode_e4m3((s << 7) | ((e - 1 + 7) << 3) | (m << 2))
        assert mx.decode_e2m1(c) == ref, c


def test_fp4_nibble_order_and_round_trip():
    assert list(mx.unpack_fp4(np.array([0x21, 0xF3], np.uint8), 4)) == [1, 2, 3, 15]
    assert list(mx.unpack_fp4(np.array([0x21, 0xF3], np.uint8), 3)) == [1, 2, 3]
    rng = np.random.default_rng(4)
    c = rng.integers(0, 16, size=(3, 5, 37)).astype(np.uint8)
    assert np.array_equal(mx.unpack_fp4(mx.pack_fp4(c), 37), c)
    assert mx.pack_fp4(np.array([7], np.uint8))[0] == 7  # odd K: high nibble 0


def _frac_e2m1(code):
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    sign = -1 if s else 1
    if e == 0:
        return sign * Fraction(m, 2)
    return sign * (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)


def test_fp4_brute_force_fractions():
    rng = np.random.default_rng(21)
    M, N, K = 3, 4, 70  # three scale blocks, the last one ragged; K even
    Ac = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    Bc = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sfa = rng.integers(118, 137, size=(M, 3)).astype(np.uint8)
    sfb = rng.integers(118, 137, size=(N, 3)).astype(np.uint8)
    got = mx.gemm_mxfp4_f64(mx.pack_fp4(Ac), mx.pack_fp4(Bc), K, sfa, sfb)
    for i in range(M):
        for j in range(N):
            exact = sum(_frac_e2m1(int(Ac[i, k])) * Fraction(2) ** (int(sfa[i, k // 32]) - 127) *
                        _frac_e2m1(int(Bc[j, k])) * Fraction(2) ** (int(sfb[j, k // 32]) - 127)
                        for k in range(K))
            assert got[i, j] == float(exact), (i, j)


def test_fp4_planted_nibble_swap_is_caught():
    """Reading the high nibble first (a plausible packing mistake) changes
    the product of a row whose two nibbles differ."""
    Ac = np.array([[1, 2] * 16], np.uint8)   # values 0.5, 1, 0.5, 1, ...
    Bc = np.array([[2, 0] * 16], np.uint8)   # values 1, 0, 1, 0, ...
    one = np.full((1, 1), 127, np.uint8)
    good = mx.gemm_mxfp4_f64(mx.pack_fp4(Ac), mx.pack_fp4(Bc), 32, one, one)
    swapped = mx.gemm_mxfp4_f64(mx.pack_fp4(Ac[:, ::-1].copy())[:, ::-1].copy(), mx.pack_fp4(Bc), 32, one, one)
    assert good[0, 0] == 16 * 0.5
    assert swapped[0, 0] != good[0, 0]
