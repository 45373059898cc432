"""GPU parity of the direct-load kernel (small problems: one CTA per 128 x 64
tile, operands copied into shared memory by the threads with plain loads).

Integer-valued bf16 inputs make every partial sum an exact fp32 integer, so
the kernel must equal the fp64 oracle bit for bit; on random floats it must
equal the persistent kernel bit for bit, because both issue the same
tcgen05 MMAs on the same shared-memory images (persistent kernel with
64-wide tiles, no K split).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev, oracle_dense

pytestmark = pytest.mark.gpu

DIRECT = dict(direct=2)
PERSISTENT_SAME_MMAS = dict(direct=1, block_n=64, split_k=1, stream_k=1)
SHAPES = [(1, 1, 1), (7, 5, 3), (17, 63, 65), (127, 129, 128), (129, 255, 257), (200, 300, 40),
          (65, 513, 191), (197, 131, 77), (256, 128, 513), (64, 64, 1000)]
LAYOUTS = [(0, 0), (0, 1), (1, 0), (1, 1)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tg.load()
    yield


def _layout(t, cm):
    """t [.., R, C] -> the same matrix stored column-major (a transposed view)."""
    return t.transpose(-1, -2).contiguous().transpose(-1, -2) if cm else t


def _gemm(A, B, C, **opts):
    tg.gemm(A, B, C, options=tg.make_options(**opts))  # the binding reads the layouts off the strides
    st = tg.device_error()
    assert st == tg.TG_OK, tg.STATUS_NAMES.get(st, st)
    return C


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nn", "nt", "tn", "tt"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_direct_exact_integer(shape, layout):
    M, N, K = shape
    A, B = synth.make_int_inputs(1, M, N, K, seed=M * 7 + N * 3 + K)
    Ad, Bd = _layout(A.to(dev()), layout[0]), _layout(B.to(dev()), layout[1])
    C = torch.full((M, N), float("nan"), device=dev())
    _gemm(Ad, Bd, C, **DIRECT)
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A, B))


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nn", "nt", "tn", "tt"])
@pytest.mark.parametrize("shape", [(197, 131, 77), (129, 65, 257), (300, 200, 1000), (128, 64, 256)],
                         ids=lambda s: "x".join(map(str, s)))
def test_direct_bitwise_equals_persistent(shape, layout):
    M, N, K = shape
    A, B = synth.make_inputs(1, M, N, K, "normal", seed=M + N + K)
    Ad, Bd = _layout(A.to(dev()), layout[0]), _layout(B.to(dev()), layout[1])
    Cd = _gemm(Ad, Bd, torch.empty(M, N, device=dev()), **DIRECT)
    Cp = _gemm(Ad, Bd, torch.empty(M, N, device=dev()), **PERSISTENT_SAME_MMAS)
    assert torch.equal(Cd, Cp)


def test_direct_batched_broadcast_and_gaps():
    """Stacked problems with gaps between them and between rows, and an
    operand shared by every problem (batch stride 0)."""
    batch, M, N, K = 5, 70, 90, 150
    A, B = synth.make_int_inputs(batch, M, N, K, seed=11)
    Abuf = torch.zeros(batch, M + 3, K + 5, dtype=torch.bfloat16, device=dev())
    Abuf[:, :M, :K] = A.to(dev())
    Ad = Abuf[:, :M, :K]
    Bd = B.to(dev())
    Cbuf = torch.full((batch, M + 2, N + 7), -3.0, device=dev())
    C = Cbuf[:, :M, :N]
    tg.gemm(Ad, Bd, C, options=tg.make_options(**DIRECT))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A, B))
    assert torch.all(Cbuf[:, M:, :] == -3.0) and torch.all(Cbuf[:, :, N:] == -3.0)
    # B shared by every problem
    B1 = B[0]
    C2 = tg.gemm(Ad, B1.to(dev()), options=tg.make_options(**DIRECT))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C2.cpu().double().numpy(), oracle_dense(A, B1.expand(batch, K, N).contiguous()))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_direct_fused_epilogue_bitwise_equals_persistent(out):
    M, N, K = 150, 100, 120
    A, B = synth.make_inputs(1, M, N, K, "normal", seed=5)
    Ad, Bd = A.to(dev()), B.to(dev())
    g = torch.Generator().manual_seed(6)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    bias = torch.randn(N, generator=g).to(dev())
    res = torch.randn(M, N, generator=g).to(dt).to(dev())
    outs = []
    for opts in (DIRECT, PERSISTENT_SAME_MMAS):
        D = tg.gemm_fused(Ad, Bd, bias=bias, residual=res, alpha=0.5, beta=-2.0, activation="gelu_tanh",
                          out_dtype=dt, options=tg.make_options(**opts))
        assert tg.device_error() == tg.TG_OK
        outs.append(D)
    assert torch.equal(outs[0], outs[1])


def test_direct_planner_choice_and_default_call():
    """The planner's own choice for a small problem with operands the TMA
    unit cannot address (odd pitches), and the default call on it."""
    M, N, K = 197, 131, 77
    info = tg.plan(M, N, K)
    assert info["direct"] == 2 and info["block_n"] == 64 and info["grid"] == 2 * 3
    assert info["pack_a"] == 0 and info["pack_b"] == 0 and info["workspace_bytes"] == 0
    A, B = synth.make_int_inputs(1, M, N, K, seed=2)
    C = tg.gemm(A.to(dev()), B.to(dev()))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A, B))


def test_direct_watchdog_reports_timeout_and_recovers():
    M, N, K = 100, 100, 100
    A, B = synth.make_int_inputs(1, M, N, K, seed=9)
    Ad, Bd = A.to(dev()), B.to(dev())
    tg.gemm(Ad, Bd, options=tg.make_options(debug_stall=1, timeout_ns=20_000_000, **DIRECT))
    assert tg.device_error() == tg.TG_ERR_TIMEOUT
    assert tg.device_error() == tg.TG_OK
    C = tg.gemm(Ad, Bd, options=tg.make_options(**DIRECT))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(A, B))


def test_direct_trace_stamps_in_order():
    M, N, K = 300, 200, 600
    A, B = synth.make_int_inputs(1, M, N, K, seed=4)
    info = tg.plan(M, N, K, options=tg.make_options(**DIRECT))
    tr = torch.zeros(info["grid"] * 8, dtype=torch.int64, device=dev())
    opts = tg.make_options(**DIRECT)
    opts.trace_buffer = tr.data_ptr()
    tg.gemm(A.to(dev()), B.to(dev()), options=opts)
    assert tg.device_error() == tg.TG_OK
    t = tr.view(-1, 8).cpu()
    assert torch.all(t[:, 0] > 0)
    for k in range(7):
        assert torch.all(t[:, k + 1] >= t[:, k]), k


@pytest.mark.parametrize("layout", LAYOUTS, ids=["nn", "nt", "tn", "tt"])
@pytest.mark.parametrize("shape", [(8, 8, 8), (128, 64, 64), (200, 136, 256), (256, 256, 512), (64, 520, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_direct_vector_staging(shape, layout):
    """Operands with 16-byte aligned pitches and extents that are multiples
    of 8 are staged in 16-byte units; the same operands with a pitch one
    element longer go element by element.  Both equal the oracle exactly."""
    M, N, K = shape
    A, B = synth.make_int_inputs(1, M, N, K, seed=M + 2 * N + 3 * K)
    want = oracle_dense(A, B)
    for pad in (0, 1):
        Ad = _layout(A.to(dev()), layout[0])
        Bd = _layout(B.to(dev()), layout[1])
        if pad:
            # the same matrices in buffers with one extra element a row (or column)
            def padded(t):
                buf = torch.zeros(t.shape[0] + (1 if t.stride(0) == 1 else 0),
                                  t.shape[1] + (1 if t.stride(1) == 1 else 0), dtype=t.dtype, device=t.device)
                if t.stride(1) == 1:
                    buf[:, :t.shape[1]] = t
                    return buf[:, :t.shape[1]]
                buf = torch.zeros(t.shape[1], t.shape[0] + 1, dtype=t.dtype, device=t.device)
                buf[:, :t.shape[0]] = t.t()
                return buf[:, :t.shape[0]].t()
            Ad, Bd = padded(Ad), padded(Bd)
        C = torch.full((M, N), float("nan"), device=dev())
        _gemm(Ad, Bd, C, **DIRECT)
        assert np.array_equal(C.cpu().double().numpy(), want), pad
