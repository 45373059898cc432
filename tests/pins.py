"""Pins for a GEMM implementation: checks that come from the mathematics and
the pages, not from any implementation.

Each ``pin_*`` takes ``gemm(A_u16, B_u16, M, N, K, lda, ldb, ldc, batch, sA,
sB, sC) -> flat float64 C`` and raises ``AssertionError`` on a mismatch.  The
oracle must pass all of them; ``tests/test_oracle.py`` also shows that
plausible mistakes (a dropped term, a sign, a transposed operand, a wrong
stride, fp32 accumulation, accumulate-into-C) each fail at least one.

Exact reference values come from ``fractions.Fraction`` arithmetic on bf16
values decoded field by field (sign, exponent, mantissa) - an independent
decoding from the oracle's bit-shift widening.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


# ---------------------------------------------------------------- helpers
def bf16_value(bits: int) -> Fraction:
    """Exact value of a bf16 pattern from its IEEE fields (finite only)."""
    sign = -1 if (bits >> 15) & 1 else 1
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    if exp == 0xFF:
        raise ValueError("non-finite bf16")
    if exp == 0:
        return sign * Fraction(man, 128) * Fraction(1, 2 ** 126)
    e = exp - 127
    v = Fraction(128 + man, 128)
    return sign * (v * 2 ** e if e >= 0 else v / 2 ** (-e))


def bf16_bits_of_int(v: int) -> int:
    """bf16 pattern of a small integer |v| <= 256 (exactly representable)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.bit_length() - 1
    man = ((a << 7) >> e) & 0x7F if e <= 7 else (a >> (e - 7)) & 0x7F
    return sign | ((e + 127) << 7) | man


def ints_to_bf16(arr) -> np.ndarray:
    a = np.asarray(arr)
    out = np.zeros(a.shape, dtype=np.uint16)
    for idx, v in np.ndenumerate(a):
        out[idx] = bf16_bits_of_int(int(v))
    return out


def exact_gemm(A: np.ndarray, B: np.ndarray, M, N, K, lda, ldb, batch, sA, sB):
    """Exact products as Fractions: list over batch of MxN nested lists."""
    dec = {}

    def val(bits):
        bits = int(bits)
        if bits not in dec:
            dec[bits] = bf16_value(bits)
        return dec[bits]

    out = []
    for b in range(batch):
        rows = []
        for i in range(M):
            row = []
            for j in range(N):
                s = Fraction(0)
                for k in range(K):
                    s += val(A[b * sA + i * lda + k]) * val(B[b * sB + k * ldb + j])
                row.append(s)
            rows.append(row)
        out.append(rows)
    return out


def dense_call(gemm, A2, B2):
    """Call ``gemm`` on dense single problems given 2-D uint16 arrays."""
    M, K = A2.shape
    K2, N = B2.shape
    assert K == K2
    c = gemm(np.ascontiguousarray(A2).reshape(-1), np.ascontiguousarray(B2).reshape(-1),
             M, N, K, K, N, N, 1, M * K, K * N, M * N)
    return np.asarray(c, dtype=np.float64).reshape(M, N)


# ---------------------------------------------------------------- pins
def pin_bruteforce_int(gemm, rng):
    """Tiny shapes, small-integer inputs: the fp64 result is exact."""
    for (M, N, K) in [(1, 1, 1), (2, 3, 4), (5, 7, 3), (8, 8, 8), (3, 1, 6), (1, 6, 2)]:
        a = rng.integers(-16, 17, size=(M, K))
        b = rng.integers(-16, 17, size=(K, N))
        c = dense_call(gemm, ints_to_bf16(a), ints_to_bf16(b))
        for i in range(M):
            for j in range(N):
                want = sum(int(a[i, k]) * int(b[k, j]) for k in range(K))
                assert c[i, j] == want, (M, N, K, i, j, c[i, j], want)


def pin_bruteforce_float(gemm, rng):
    """Tiny shapes, random finite bf16 floats of mixed magnitude: the fp64
    result is within the textbook summation bound of the exact rational sum,
    |fl(s) - s| <= gamma_K * sum |a_k b_k| with gamma_K = K u / (1 - K u),
    u = 2^-53 (products of two bf16 are exact in fp64)."""
    u = Fraction(1, 2 ** 53)
    for (M, N, K) in [(2, 3, 5), (4, 4, 8), (7, 2, 6), (1, 5, 7)]:
        a = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-12, 12, (M, K)))).astype(np.float32)
        b = (rng.standard_normal((K, N)) * np.exp2(rng.integers(-12, 12, (K, N)))).astype(np.float32)
        abits = (a.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16 (any bf16 will do)
        bbits = (b.view(np.uint32) >> 16).astype(np.uint16)
        c = dense_call(gemm, abits, bbits)
        ex = exact_gemm(abits.reshape(-1), bbits.reshape(-1), M, N, K, K, N, 1, 0, 0)[0]
        gamma = K * u / (1 - K * u)
        for i in range(M):
            for j in range(N):
                mag = sum(abs(bf16_value(int(abits[i, k])) * bf16_value(int(bbits[k, j]))) for k in range(K))
                err = abs(Fraction(float(c[i, j])) - ex[i][j])
                assert err <= gamma * mag, (M, N, K, i, j, float(err), float(gamma * mag))


def pin_identity(gemm, rng):
    """A = I (and A = [I; 0]) gives C = B exactly."""
    for (M, K, N) in [(6, 6, 9), (9, 5, 4)]:
        ident = np.zeros((M, K), dtype=np.int64)
        for t in range(min(M, K)):
            ident[t, t] = 1
        b = rng.integers(-100, 101, size=(K, N))
        c = dense_call(gemm, ints_to_bf16(ident), ints_to_bf16(b))
        want = np.zeros((M, N))
        want[: min(M, K)] = b[: min(M, K)]
        assert np.array_equal(c, want), "identity"


def pin_permutation(gemm, rng):
    """C = P B permutes the rows of B; C = A Q permutes the columns of A."""
    M = K = 7
    N = 5
    perm = rng.permutation(M)
    P = np.zeros((M, K), dtype=np.int64)
    P[np.arange(M), perm] = 1
    b = rng.integers(-50, 51, size=(K, N))
    c = dense_call(gemm, ints_to_bf16(P), ints_to_bf16(b))
    assert np.array_equal(c, b[perm].astype(np.float64)), "row permutation"
    # right multiplication: A (4 x 6) times Q (6 x 6) moves column q to perm2[q]
    a = rng.integers(-50, 51, size=(4, 6))
    perm2 = rng.permutation(6)
    Q = np.zeros((6, 6), dtype=np.int64)
    Q[np.arange(6), perm2] = 1
    c2 = dense_call(gemm, ints_to_bf16(a), ints_to_bf16(Q))
    want = np.zeros((4, 6))
    want[:, perm2] = a
    assert np.array_equal(c2, want), "column permutation"


def pin_all_ones(gemm, rng):
    """All-ones A and B: every entry of C equals K exactly."""
    for (M, N, K) in [(3, 4, 1), (5, 3, 777), (2, 2, 5000)]:
        one = bf16_bits_of_int(1)
        a = np.full((M, K), one, dtype=np.uint16)
        b = np.full((K, N), one, dtype=np.uint16)
        c = dense_call(gemm, a, b)
        assert np.all(c == K), ("all-ones", M, N, K)


def pin_pad_invariance(gemm, rng):
    """OCANNL "Module Ir.Schedule", Pad-to-tile: padding the extents with
    zero rows/columns leaves the valid block of C unchanged (exact)."""
    M, N, K = 5, 6, 7
    a = rng.integers(-9, 10, size=(M, K))
    b = rng.integers(-9, 10, size=(K, N))
    base = dense_call(gemm, ints_to_bf16(a), ints_to_bf16(b))
    Mp, Np, Kp = 8, 16, 16
    ap = np.zeros((Mp, Kp), dtype=np.int64)
    bp = np.zeros((Kp, Np), dtype=np.int64)
    ap[:M, :K] = a
    bp[:K, :N] = b
    # junk in the padded rows of A / columns of B must not leak into the block
    ap[M:, :K] = 3
    bp[:K, N:] = -2
    padded = dense_call(gemm, ints_to_bf16(ap), ints_to_bf16(bp))
    assert np.array_equal(padded[:M, :N], base), "pad invariance"
    want = np.array([[sum(int(a[i, k]) * int(b[k, j]) for k in range(K)) for j in range(N)] for i in range(M)])
    assert np.array_equal(base, want.astype(np.float64)), "pad base"


def pin_split_invariance(gemm, rng):
    """OCANNL "Module Ir.Schedule", two-pass split reduction: the sum of the
    partial products over consecutive K chunks equals the full product
    (exact with integer inputs)."""
    M, N, K = 4, 5, 23
    a = rng.integers(-9, 10, size=(M, K))
    b = rng.integers(-9, 10, size=(K, N))
    full = dense_call(gemm, ints_to_bf16(a), ints_to_bf16(b))
    for chunks in (2, 3, 5):
        bounds = [(s * K) // chunks for s in range(chunks + 1)]
        total = np.zeros((M, N))
        for s in range(chunks):
            k0, k1 = bounds[s], bounds[s + 1]
            total += dense_call(gemm, ints_to_bf16(a[:, k0:k1]), ints_to_bf16(b[k0:k1]))
        assert np.array_equal(total, full), ("split", chunks)


def pin_strided_batched(gemm, rng):
    """batch > 1 with ld > extent and gaps between problems: each problem
    equals its own brute-force product, and gaps in C stay untouched (0)."""
    batch, M, N, K = 3, 4, 5, 6
    lda, ldb, ldc = K + 3, N + 2, N + 4
    sA, sB, sC = M * lda + 5, K * ldb + 7, M * ldc + 3
    A = np.zeros(batch * sA, dtype=np.uint16)
    B = np.zeros(batch * sB, dtype=np.uint16)
    vals_a = rng.integers(-9, 10, size=(batch, M, K))
    vals_b = rng.integers(-9, 10, size=(batch, K, N))
    junk = bf16_bits_of_int(77)
    A[:] = junk
    B[:] = junk
    for bb in range(batch):
        for i in range(M):
            A[bb * sA + i * lda: bb * sA + i * lda + K] = ints_to_bf16(vals_a[bb, i])
        for k in range(K):
            B[bb * sB + k * ldb: bb * sB + k * ldb + N] = ints_to_bf16(vals_b[bb, k])
    c = np.asarray(gemm(A, B, M, N, K, lda, ldb, ldc, batch, sA, sB, sC), dtype=np.float64)
    written = np.zeros(c.shape, dtype=bool)
    for bb in range(batch):
        for i in range(M):
            for j in range(N):
                want = sum(int(vals_a[bb, i, k]) * int(vals_b[bb, k, j]) for k in range(K))
                pos = bb * sC + i * ldc + j
                assert c[pos] == want, ("strided", bb, i, j, c[pos], want)
                written[pos] = True
    assert np.all(c[~written] == 0), "gap elements of C were written"


ALL_PINS = [pin_bruteforce_int, pin_bruteforce_float, pin_identity, pin_permutation,
            pin_all_ones, pin_pad_invariance, pin_split_invariance, pin_strided_batched]
