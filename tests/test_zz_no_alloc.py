"""The non-allocating split-K entry point (tg_gemm_splitk_static) against the
allocating one (tg_gemm_ex with the same split factor), through the C ABI.

Callers that cannot allocate device memory - plugins inside a framework
whose memory pool owns the GPU, services that may not call cudaMalloc after
start-up - use tg_gemm_splitk_static; its scratch is a static device array
that every call shares.  Two calls in a row check that leftover contents of
that array from the first call do not leak into the second.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import assert_close, oracle_dense

pytestmark = pytest.mark.gpu


def _call_static(A, B, C, split_k):
    M, K = A.shape
    N = B.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return tg.tg_gemm_splitk_static(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N, 1,
                                    M * K, K * N, M * N, split_k, stream)


def _call_ex(A, B, C, split_k):
    M, K = A.shape
    N = B.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return tg.tg_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, K, N, N, 1, M * K, K * N,
                         M * N, stream, tg.make_options(split_k=split_k))


def test_static_scratch_entry_matches_allocating_entry_twice():
    tg.load()
    dev = torch.device("cuda:0")
    split_k = 4
    shapes = [(64, 2048, 4096, "normal002", 1), (200, 640, 1000, "uniform", 2)]
    for call in range(2):  # two calls in a row share (and reuse) the static array
        for (M, N, K, dist, seed) in shapes:
            A_cpu, B_cpu = synth.make_inputs(1, M, N, K, dist, seed=seed + 10 * call)
            A, B = A_cpu.to(dev), B_cpu.to(dev)
            C_static = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
            C_ex = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
            assert _call_static(A, B, C_static, split_k) == tg.TG_OK
            assert _call_ex(A, B, C_ex, split_k) == tg.TG_OK
            torch.cuda.synchronize()
            assert tg.device_error() == tg.TG_OK
            got = C_static.cpu().double().numpy()
            ref = C_ex.cpu().double().numpy()
            assert_close(got, ref, K, f"call {call} {M}x{N}x{K}")
            assert_close(got, oracle_dense(A_cpu, B_cpu), K, f"call {call} vs oracle")


def test_static_scratch_entry_rejects_oversize():
    tg.load()
    dev = torch.device("cuda:0")
    # 64 x 28672 with 16 splits needs far more than the 16 MiB of partial tiles
    M, N, K = 64, 28672, 8192
    A = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(K, N, dtype=torch.bfloat16, device=dev)
    C = torch.zeros(M, N, dtype=torch.float32, device=dev)
    assert _call_static(A, B, C, 16) == tg.TG_ERR_UNSUPPORTED
    assert _call_static(A, B, C, 0) == tg.TG_ERR_INVALID_ARG
    assert np.all(C.cpu().numpy() == 0)
