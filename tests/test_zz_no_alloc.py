"""The non-allocating split-K entry point (tg_gemm_splitk_static) against the
allocating one (tg_gemm_ex with the same split factor), through the C ABI.

Callers that cannot allocate device memory - plugins inside a framework
whose memory pool owns the GPU, services that may not call cudaMalloc after
start-up - use tg_gemm_splitk_static; its scratch is a static device array
that every call shares.  Two calls in a row check that leftover contents of
that array from the first call do not leak into the second.  The watchdog of
that entry point reports through tg_device_error() like the others; its
rejections (sizes past the array, operands that would need a pack copy) are
checked, and so is that a warmed-up call allocates no device memory.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import assert_close, oracle_dense

pytestmark = pytest.mark.gpu


def _dense_args(A, B, C):
    """(M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC) of dense
    [batch?, M, K] x [batch?, K, N] -> [batch?, M, N] tensors."""
    batch = A.shape[0] if A.dim() == 3 else 1
    M, K = A.shape[-2:]
    N = B.shape[-1]
    return M, N, K, K, N, N, batch, M * K, K * N, M * N


def _call_static(A, B, C, split_k, lda=None):
    M, N, K, lda0, ldb, ldc, batch, sA, sB, sC = _dense_args(A, B, C)
    stream = torch.cuda.current_stream().cuda_stream
    return tg.tg_gemm_splitk_static(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                    lda0 if lda is None else lda, ldb, ldc, batch, sA, sB, sC,
                                    split_k, stream)


def _call_ex(A, B, C, split_k):
    M, N, K, lda, ldb, ldc, batch, sA, sB, sC = _dense_args(A, B, C)
    stream = torch.cuda.current_stream().cuda_stream
    return tg.tg_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, ldc, batch, sA, sB,
                         sC, stream, tg.make_options(split_k=split_k))


def _both(A_cpu, B_cpu, split_k, what):
    dev = torch.device("cuda:0")
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    shape = tuple(A.shape[:-1]) + (B.shape[-1],)
    C_static = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
    C_ex = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
    assert _call_static(A, B, C_static, split_k) == tg.TG_OK, what
    assert _call_ex(A, B, C_ex, split_k) == tg.TG_OK, what
    torch.cuda.synchronize()
    assert tg.device_error() == tg.TG_OK, what
    got = C_static.cpu().double().numpy()
    ref = C_ex.cpu().double().numpy()
    K = A.shape[-1]
    assert_close(got, ref, K, f"{what} vs tg_gemm_ex")
    assert_close(got, oracle_dense(A_cpu, B_cpu), K, f"{what} vs oracle")
    return got


def test_static_scratch_entry_matches_allocating_entry_twice():
    tg.load()
    split_k = 4
    shapes = [(64, 2048, 4096, "normal002", 1), (200, 640, 1000, "uniform", 2)]
    for call in range(2):  # two calls in a row share (and reuse) the static array
        for (M, N, K, dist, seed) in shapes:
            A_cpu, B_cpu = synth.make_inputs(1, M, N, K, dist, seed=seed + 10 * call)
            _both(A_cpu, B_cpu, split_k, f"call {call} {M}x{N}x{K}")


def test_static_scratch_entry_batched_and_ragged():
    """A batch of problems, and extents off every tile multiple (masked
    fringe rows and columns, a K tail), each at two split factors; integer
    inputs must match the oracle bit for bit.  (Rows of A and B stay 16-byte
    aligned - K and N multiples of 8 - since this entry point has no pack
    copy.)"""
    tg.load()
    for split_k in (2, 3):
        A_cpu, B_cpu = synth.make_inputs(6, 150, 296, 704, "uniform", seed=30 + split_k)
        _both(A_cpu, B_cpu, split_k, f"batched split {split_k}")
        A_cpu, B_cpu = synth.make_inputs(1, 257, 200, 1000, "normal", seed=40 + split_k)
        _both(A_cpu, B_cpu, split_k, f"ragged split {split_k}")
        Ai, Bi = synth.make_int_inputs(3, 131, 72, 520, seed=50 + split_k)
        got = _both(Ai, Bi, split_k, f"integer split {split_k}")
        assert np.array_equal(got, oracle_dense(Ai, Bi))


def test_static_scratch_entry_watchdog_reports_timeout():
    """The self-test stall makes the kernel's wait expire; the expiry lands in
    the static array's error word, tg_device_error() reports it once and
    clears it, and the next call is exact."""
    tg.load()
    dev = torch.device("cuda:0")
    Ai, Bi = synth.make_int_inputs(1, 200, 296, 1024, seed=61)
    A, B = Ai.to(dev), Bi.to(dev)
    C = torch.zeros(200, 296, dtype=torch.float32, device=dev)
    os.environ["TG_DEBUG_STALL_NS"] = "20000000"  # 20 ms
    try:
        assert _call_static(A, B, C, 4) == tg.TG_OK
    finally:
        del os.environ["TG_DEBUG_STALL_NS"]
    assert tg.device_error() == tg.TG_ERR_TIMEOUT
    assert tg.device_error() == tg.TG_OK
    C.fill_(float("nan"))
    assert _call_static(A, B, C, 4) == tg.TG_OK
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(Ai, Bi))


def test_static_scratch_entry_rejects_oversize_and_misaligned():
    tg.load()
    dev = torch.device("cuda:0")
    # 64 x 28672 with 16 splits needs far more than the 16 MiB of partial tiles
    M, N, K = 64, 28672, 8192
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(K, N, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(M, N, dtype=torch.float32, device=dev)
    assert _call_static(A, B, C, 16) == tg.TG_ERR_UNSUPPORTED
    assert _call_static(A, B, C, 0) == tg.TG_ERR_INVALID_ARG
    # more output tiles than the array has counters (4097 one-tile problems)
    Ab = torch.zeros(4097, 8, 64, dtype=torch.bfloat16, device=dev)
    Bb = torch.zeros(4097, 64, 8, dtype=torch.bfloat16, device=dev)
    Cb = torch.zeros(4097, 8, 8, dtype=torch.float32, device=dev)
    assert _call_static(Ab, Bb, Cb, 1) == tg.TG_ERR_UNSUPPORTED
    # rows of A 2 bytes off a 16-byte multiple: would need the pack copy
    Am = torch.zeros(M, K + 1, dtype=torch.bfloat16, device=dev)[:, :K]
    assert _call_static(Am, B, C, 2, lda=K + 1) == tg.TG_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert np.all(C.cpu().numpy() == 0)
    assert np.all(Cb.cpu().numpy() == 0)


def test_static_scratch_entry_allocates_nothing():
    """After one warmed-up call, further calls leave the device's free memory
    unchanged (the library takes nothing from the device allocator)."""
    tg.load()
    dev = torch.device("cuda:0")
    A_cpu, B_cpu = synth.make_inputs(2, 256, 512, 2048, "uniform", seed=71)
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    C = torch.empty(2, 256, 512, dtype=torch.float32, device=dev)
    assert _call_static(A, B, C, 4) == tg.TG_OK
    assert tg.device_error() == tg.TG_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        assert _call_static(A, B, C, 4) == tg.TG_OK
        assert tg.device_error() == tg.TG_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, (free0, free1)
    assert_close(C.cpu().double().numpy(), oracle_dense(A_cpu, B_cpu), 2048, "after the no-allocation calls")
