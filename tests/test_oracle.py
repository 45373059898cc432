"""The oracle against its pins (CPU only).

The oracle (``oracle/gemm_f64.c``) is pinned by:
* exact brute force on tiny shapes (integers, and rationals for floats),
* closed forms: identity, permutations, all-ones (C = K),
* the pages' invariants: pad-to-tile and split-reduction invariance,
* strided / batched addressing with guard gaps,
and the pins are shown to be sharp: each plausible mistake planted in a
CPU stand-in of the oracle fails at least one pin.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import pins
import synth


def oracle_call(A, B, M, N, K, lda, ldb, ldc, batch, sA, sB, sC):
    return oracle.gemm_f64(A, B, M, N, K, lda, ldb, ldc, batch, sA, sB, sC)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    pin(oracle_call, np.random.default_rng(1234))


# ------------------------------------------------------------ planted mistakes
def _widen(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _py_gemm(A, B, M, N, K, lda, ldb, ldc, batch, sA, sB, sC, mistake=None):
    """A CPU stand-in for the oracle with one planted mistake."""
    a = _widen(A)
    b = _widen(B)
    c = np.zeros(batch * sC)
    acc_t = np.float32 if mistake == "fp32_accumulate" else np.float64
    for bb in range(batch):
        for i in range(M):
            for j in range(N):
                s = acc_t(1.0) if mistake == "accumulate_into_c" else acc_t(0.0)
                kmax = K - 1 if mistake == "drop_last_term" else K
                for k in range(kmax):
                    row_stride = K if mistake == "ignore_lda" else lda
                    bstride = M * K if mistake == "ignore_batch_stride" else sA
                    av = a[(bb * bstride + i * row_stride + k) % a.size]
                    if mistake == "transpose_b":
                        bv = b[(bb * sB + j * ldb + k) % b.size]
                    else:
                        bv = b[bb * sB + k * ldb + j]
                    t = acc_t(av) * acc_t(bv)
                    if mistake == "sign" and k == 0:
                        t = -t
                    s = acc_t(s + t)
                if mistake == "transpose_c" and i < N and j < M:
                    c[bb * sC + j * ldc + i] = s
                else:
                    c[bb * sC + i * ldc + j] = s
    return c


MISTAKES = ["transpose_b", "drop_last_term", "sign", "fp32_accumulate", "ignore_lda",
            "ignore_batch_stride", "accumulate_into_c", "transpose_c"]


def test_pins_accept_a_correct_stand_in():
    """Control: the mistake-free stand-in passes every pin (the pins are not
    stricter than the mathematics)."""
    for pin in pins.ALL_PINS:
        pin(lambda *args: _py_gemm(*args), np.random.default_rng(1234))


@pytest.mark.parametrize("mistake", MISTAKES)
def test_pins_catch_planted_mistake(mistake):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lambda *args: _py_gemm(*args, mistake=mistake), np.random.default_rng(1234))
        except AssertionError:
            failed.append(pin.__name__)
        except (IndexError, ValueError):
            failed.append(pin.__name__ + "(crash)")
    assert failed, f"no pin catches the planted mistake {mistake!r}"


# ------------------------------------------------------------ entries form
def test_entries_match_exact_rationals():
    """The dot-product form for sampled entries is exact-within-bound against
    Fraction arithmetic on a seeded workload of the ragged small shape."""
    w = synth.WORKLOADS["ragged_197x131x77"]
    A, B = synth.workload_inputs(w)
    a = synth.bits_u16(A).reshape(-1)
    b = synth.bits_u16(B).reshape(-1)
    bi, ii, jj = synth.sample_indices(1, w.M, w.N, 40, seed=5)
    got = oracle.gemm_entries_f64(a, b, w.M, w.N, w.K, bi, ii, jj)
    u = Fraction(1, 2 ** 53)
    gamma = w.K * u / (1 - w.K * u)
    for t in range(len(bi)):
        i, j = int(ii[t]), int(jj[t])
        terms = [pins.bf16_value(int(a[i * w.K + k])) * pins.bf16_value(int(b[k * w.N + j]))
                 for k in range(w.K)]
        exact = sum(terms, Fraction(0))
        mag = sum((abs(x) for x in terms), Fraction(0))
        assert abs(Fraction(float(got[t])) - exact) <= gamma * mag


def test_entries_equal_full_product():
    """Both forms sum k in ascending order, so sampled entries equal the full
    product's entries bit for bit (batched, strided)."""
    batch, M, N, K = 3, 37, 29, 53
    A, B = synth.make_inputs(batch, M, N, K, "normal", seed=9)
    full = oracle.gemm_dense_f64(A, B)
    bi, ii, jj = synth.sample_indices(batch, M, N, 200, seed=1, tile_m=16, tile_n=16)
    ent = oracle.gemm_entries_f64(A, B, M, N, K, bi, ii, jj, batch=batch)
    assert np.array_equal(ent, full[bi, ii, jj])


def test_entries_reject_out_of_range():
    A, B = synth.make_inputs(1, 4, 4, 4, "uniform", seed=0)
    with pytest.raises(ValueError):
        oracle.gemm_entries_f64(A, B, 4, 4, 4, [0], [4], [0])


def test_zero_k_gives_zeros():
    """An empty reduction is the additive identity."""
    a = np.zeros(0, dtype=np.uint16)
    b = np.zeros(0, dtype=np.uint16)
    c = oracle.gemm_f64(a, b, 3, 4, 0)
    assert np.array_equal(c, np.zeros(12))


def test_oracle_rejects_bad_strides():
    A, B = synth.make_inputs(1, 4, 4, 4, "uniform", seed=0)
    with pytest.raises(ValueError):
        oracle.gemm_f64(A, B, 4, 4, 4, lda=3)


def test_thread_count_independent():
    """Each row's sum order is fixed, so the result does not depend on how
    OpenMP splits rows: compare a batched product with per-problem calls."""
    batch, M, N, K = 4, 33, 17, 45
    A, B = synth.make_inputs(batch, M, N, K, "uniform", seed=3)
    full = oracle.gemm_dense_f64(A, B)
    for bb in range(batch):
        one = oracle.gemm_dense_f64(A[bb], B[bb])
        assert np.array_equal(one, full[bb])


def test_seeded_inputs_reproducible():
    """The generator recipe is deterministic and draws A before B."""
    a1, b1 = synth.make_inputs(1, 8, 6, 5, "uniform", seed=7)
    a2, b2 = synth.make_inputs(1, 8, 6, 5, "uniform", seed=7)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)
    gen = torch.Generator("cpu").manual_seed(7)
    a3 = (torch.rand((1, 8, 5), generator=gen) * 2 - 1).to(torch.bfloat16)[0]
    assert torch.equal(a1, a3)
    ai, bi = synth.make_int_inputs(1, 8, 6, 4096, seed=1)
    assert float(ai.float().abs().max()) <= synth.int_magnitude(4096)
    assert synth.int_magnitude(4096) ** 2 * 4096 < 2 ** 24


def test_workload_recipe():
    w = synth.WORKLOADS["skinny_64x28672x8192"]
    assert (w.batch, w.M, w.N, w.K, w.seed) == (1, 64, 28672, 8192, 4)
    assert synth.WORKLOADS["square_4096"].flops == 2 * 4096 ** 3
    assert synth.WORKLOADS["batched_64x384x640x1000"].bytes_moved == 193_986_560
