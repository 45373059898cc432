"""CUDA graph capture of library calls: after one warm-up call (which sizes
the stream's workspaces and sets the kernels' attributes), a call enqueues
only kernel launches, so it can be captured in a CUDA graph and replayed;
each replay reads the operands' current contents.  Checked for the
persistent kernel (plain, packed operands, split-K and stream-K, whose tile
counters the kernel itself returns to zero), the direct-load kernel and
the fused epilogue."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev, oracle_dense

pytestmark = pytest.mark.gpu

CASES = [
    ("persistent", (300, 520, 640), dict(direct=1)),
    ("packed", (197, 131, 300), dict(direct=1)),
    ("split_k", (128, 256, 2048), dict(direct=1, block_n=128, split_k=4)),
    ("stream_k", (1536, 2048, 1024), dict(direct=1, stream_k=2)),
    ("stream_k_pair", (4096, 4096, 1024), dict(direct=1, stream_k=2)),
    ("direct", (197, 131, 77), dict(direct=2)),
    ("direct_vec", (256, 256, 512), dict(direct=2)),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tg.load()
    yield


@pytest.mark.parametrize("name,shape,opts", CASES, ids=[c[0] for c in CASES])
def test_graph_capture_and_replay(name, shape, opts):
    M, N, K = shape
    o = tg.make_options(**opts)
    A0, B0 = synth.make_int_inputs(1, M, N, K, seed=M + N)
    A = A0.to(dev())
    B = B0.to(dev())
    C = torch.full((M, N), float("nan"), device=dev())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tg.gemm(A, B, C, options=o, stream=s)  # warm-up on the capturing stream
    s.synchronize()
    assert tg.device_error(s) == tg.TG_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.gemm(A, B, C, options=o, stream=s)
    for seed in (1, 2, 3):
        A1, B1 = synth.make_int_inputs(1, M, N, K, seed=seed * 101 + M)
        A.copy_(A1.to(dev()))
        B.copy_(B1.to(dev()))
        C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert tg.device_error(s) == tg.TG_OK
        assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A1, B1)), (name, seed)


def test_graph_of_a_fused_epilogue_call():
    M, N, K = 150, 100, 120
    A0, B0 = synth.make_int_inputs(1, M, N, K, seed=4)
    A, B = A0.to(dev()), B0.to(dev())
    bias = torch.arange(N, dtype=torch.float32, device=dev())
    D = torch.empty(M, N, device=dev())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tg.gemm_fused(A, B, D, bias=bias, activation="relu", stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.gemm_fused(A, B, D, bias=bias, activation="relu", stream=s)
    A1, B1 = synth.make_int_inputs(1, M, N, K, seed=5)
    A.copy_(A1.to(dev()))
    B.copy_(B1.to(dev()))
    g.replay()
    torch.cuda.synchronize()
    assert tg.device_error(s) == tg.TG_OK
    want = np.maximum(oracle_dense(A1, B1) + np.arange(N, dtype=np.float64), 0.0)
    assert np.array_equal(D.cpu().double().numpy(), want)
