"""Pins of the 8-bit floating-point oracle (CPU only).

The decoders are checked against an independent decoder (PyTorch's float8
dtypes), the OFP8 specification's named values, and exact fractions; each
planted mistake below must be caught by at least one of these pins."""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8

TORCH_DTYPES = {fp8.E4M3: torch.float8_e4m3fn, fp8.E5M2: torch.float8_e5m2}


def _torch_table(fmt):
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(TORCH_DTYPES[fmt]).to(torch.float64).numpy()


def _same(a, b):
    """Equal as values, NaN where the other is NaN, signed zeros equal in sign."""
    a, b = np.asarray(a), np.asarray(b)
    nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(nan | eq))


@pytest.mark.parametrize("fmt", [fp8.E4M3, fp8.E5M2])
def test_every_code_matches_independent_decoder(fmt):
    assert _same(fp8.table(fmt), _torch_table(fmt))


def test_e4m3_named_values():
    d = fp8.decode_e4m3
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0          # largest finite
    assert d(0x08) == 2.0 ** -6                             # smallest normal
    assert d(0x01) == 2.0 ** -9                             # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9                         # largest subnormal
    assert d(0x38) == 1.0 and d(0x40) == 2.0
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    # no infinities, and exactly two NaN codes
    t = fp8.table(fp8.E4M3)
    assert not np.any(np.isinf(t)) and int(np.isnan(t).sum()) == 2


def test_e5m2_named_values():
    d = fp8.decode_e5m2
    assert d(0x7B) == 57344.0                               # largest finite
    assert d(0x04) == 2.0 ** -14                            # smallest normal
    assert d(0x01) == 2.0 ** -16                            # smallest subnormal
    assert d(0x3C) == 1.0
    assert d(0x7C) == math.inf and d(0xFC) == -math.inf
    assert all(math.isnan(d(c)) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))


def test_integers_up_to_the_exact_range():
    """E4M3 holds every integer |n| <= 16, E5M2 every |n| <= 8 (the test
    inputs of the exact GPU cases)."""
    for fmt, top in ((fp8.E4M3, 16), (fp8.E5M2, 8)):
        vals = set(fp8.table(fmt)[np.isfinite(fp8.table(fmt))].tolist())
        assert all(float(n) in vals for n in range(-top, top + 1))


def _frac_value(fmt, code):
    """Exact value from the bit fields, in rational arithmetic."""
    if fmt == fp8.E4M3:
        s, e, m, bias, mb = code >> 7, (code >> 3) & 15, code & 7, 7, 3
    else:
        s, e, m, bias, mb = code >> 7, (code >> 2) & 31, code & 3, 15, 2
    sign = -1 if s else 1
    if e == 0:
        return sign * Fraction(m, 1 << mb) * Fraction(2) ** (1 - bias)
    return sign * (1 + Fraction(m, 1 << mb)) * Fraction(2) ** (e - bias)


def _finite_codes(fmt, rng, shape):
    t = fp8.table(fmt)
    ok = np.flatnonzero(np.isfinite(t))
    return rng.choice(ok, size=shape).astype(np.uint8)


@pytest.mark.parametrize("fa,fb", [(fp8.E4M3, fp8.E4M3), (fp8.E5M2, fp8.E4M3), (fp8.E5M2, fp8.E5M2)])
def test_gemm_brute_force_fractions(fa, fb):
    rng = np.random.default_rng(fa * 2 + fb)
    M, N, K = 3, 4, 5
    A = _finite_codes(fa, rng, (M, K))
    Bt = _finite_codes(fb, rng, (N, K))
    got = fp8.gemm_fp8_f64(A, Bt, fa, fb)
    for i in range(M):
        for j in range(N):
            exact = sum(_frac_value(fa, int(A[i, k])) * _frac_value(fb, int(Bt[j, k])) for k in range(K))
            assert got[i, j] == float(exact), (i, j)


def test_gemm_batched_and_epilogue():
    rng = np.random.default_rng(7)
    A = _finite_codes(fp8.E4M3, rng, (2, 6, 8))
    Bt = _finite_codes(fp8.E4M3, rng, (2, 5, 8))
    C = fp8.gemm_fp8_f64(A, Bt, fp8.E4M3, fp8.E4M3)
    for b in range(2):
        assert np.array_equal(C[b], fp8.decode(A[b], 0) @ fp8.decode(Bt[b], 0).T)
    D = fp8.gemm_fp8_epilogue_f64(A, Bt, 0, 0, alpha=0.5, act=1)
    assert np.array_equal(D, np.maximum(0.5 * C, 0.0))


# ---------------------------------------------------------------- planted mistakes
def _e4m3_bias8(code):
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m / 8.0, -7)
    return s * math.ldexp(1.0 + m / 8.0, e - 8)


def _e5m2_no_subnormals(code):
    v = fp8.decode_e5m2(code)
    return 0.0 if ((code >> 2) & 0x1F) == 0 else v


@pytest.mark.parametrize("fmt,bad", [(fp8.E4M3, _e4m3_bias8), (fp8.E5M2, _e5m2_no_subnormals),
                                     (fp8.E4M3, fp8.decode_e5m2), (fp8.E5M2, fp8.decode_e4m3)])
def test_planted_decoder_mistakes_are_caught(fmt, bad):
    planted = np.array([bad(c) for c in range(256)], dtype=np.float64)
    assert not _same(planted, _torch_table(fmt))
