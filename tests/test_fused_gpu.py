"""GPU parity of the fused epilogue (tg_gemm_fused), through the C ABI.

OCANNL "Module Ir.Schedule", Epilogue fusion: folding the elementwise tail
into the store-back never reorders the reduction, so the fused result equals
the two-pass form bit for bit.  Here the two-pass form is tg_gemm's fp32
output (same plan, so the same accumulation order) followed by the epilogue
formula evaluated in fp32 on the host, one rounding per operation; a bf16 D
is that value rounded to nearest even.  Transcendental activations (gelu,
silu) are compared with the fp64 oracle within a tolerance instead.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev
from oracle import epilogue as ep_oracle

pytestmark = pytest.mark.gpu

PLANS = [
    dict(block_n=128, cta_pair=1),
    dict(block_n=256, cta_pair=2, stream_k=2, max_ctas=10),
    dict(block_n=128, cta_pair=1, split_k=3),
    dict(block_n=192, cta_pair=1, epilogue=2),
    dict(direct=2),  # the direct-load kernel: batched, per-problem bias
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tg.load()
    yield


def _host_epilogue_f32(C, alpha, bias, act, beta, R):
    """The epilogue in fp32, one IEEE rounding per operation."""
    f = np.float32
    x = (f(alpha) * C.astype(np.float32)).astype(np.float32)
    if bias is not None:
        x = (x + bias.astype(np.float32)[..., None, :] if bias.ndim == 2 else x + bias.astype(np.float32)).astype(np.float32)
    if act == "relu":
        x = np.maximum(x, f(0))
    if R is not None:
        x = (x + (f(beta) * R.astype(np.float32)).astype(np.float32)).astype(np.float32)
    return x


def _to_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


@pytest.mark.parametrize("plan", PLANS, ids=lambda d: "-".join(f"{k}{v}" for k, v in d.items()))
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_fused_equals_two_pass_bitwise(plan, out, act):
    batch, M, N, K = 2, 300, 520, 700
    A, B = synth.make_inputs(batch, M, N, K, "normal", seed=5)
    gen = torch.Generator("cpu").manual_seed(9)
    bias = torch.randn(batch, N, generator=gen)
    R32 = torch.randn(batch, M, N, generator=gen)
    out_dt = torch.bfloat16 if out == "bf16" else torch.float32
    R = R32.to(out_dt)
    opts = tg.make_options(**plan)
    Ad, Bd = A.to(dev()), B.to(dev())
    D = tg.gemm_fused(Ad, Bd, bias=bias.to(dev()), residual=R.to(dev()), alpha=0.75, beta=-1.5,
                      activation=act, out_dtype=out_dt, options=opts)
    assert tg.device_error() == tg.TG_OK
    C = tg.gemm(Ad, Bd, options=opts).cpu().numpy()
    want = _host_epilogue_f32(C, 0.75, bias.numpy(), act, -1.5, R.float().numpy())
    got = D.cpu()
    if out == "bf16":
        assert torch.equal(got.view(torch.int16), _to_bf16(want).view(torch.int16))
    else:
        assert np.array_equal(got.numpy(), want)


@pytest.mark.parametrize("act", ["none", "relu", "gelu_tanh", "silu"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fused_against_oracle(act, out):
    M, N, K = 257, 389, 512
    A, B = synth.make_inputs(1, M, N, K, "uniform", seed=13)
    gen = torch.Generator("cpu").manual_seed(3)
    bias = torch.randn(N, generator=gen)
    out_dt = torch.bfloat16 if out == "bf16" else torch.float32
    R = torch.randn(M, N, generator=gen).to(out_dt)
    D = tg.gemm_fused(A.to(dev()), B.to(dev()), bias=bias.to(dev()), residual=R.to(dev()), alpha=1.25,
                      beta=0.5, activation=act, out_dtype=out_dt)
    assert tg.device_error() == tg.TG_OK
    C64 = oracle.gemm_dense_f64(A, B)
    ref = ep_oracle.apply_epilogue_f64(C64, alpha=1.25, bias=bias.double().numpy(),
                                      act=ep_oracle.ACTIVATIONS[act], beta=0.5,
                                      residual=R.double().numpy())
    got = D.double().cpu().numpy()
    # accumulation error (the GEMM contract) carried through an activation
    # with slope <= 1.2, plus fp32 rounding of the tail, plus bf16 rounding
    tol = 1.2 * 1.25 * 1e-5 * np.sqrt(K) * np.abs(C64).max() + 4e-6 * np.abs(ref)
    if out == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= tol + 1e-30), np.max(np.abs(got - ref) - tol)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fused_k_zero(out):
    """The empty sum: D = act(bias) + beta * R."""
    M, N = 33, 70
    gen = torch.Generator("cpu").manual_seed(1)
    bias = torch.randn(N, generator=gen)
    out_dt = torch.bfloat16 if out == "bf16" else torch.float32
    R = torch.randn(M, N, generator=gen).to(out_dt)
    A = torch.empty(M, 0, dtype=torch.bfloat16, device=dev())
    B = torch.empty(0, N, dtype=torch.bfloat16, device=dev())
    D = tg.gemm_fused(A, B, bias=bias.to(dev()), residual=R.to(dev()), beta=2.0, activation="relu",
                      out_dtype=out_dt)
    assert tg.device_error() == tg.TG_OK
    want = _host_epilogue_f32(np.zeros((M, N), np.float32), 1.0, bias.numpy(), "relu", 2.0, R.float().numpy())
    if out == "bf16":
        assert torch.equal(D.cpu().view(torch.int16), _to_bf16(want).view(torch.int16))
    else:
        assert np.array_equal(D.cpu().numpy(), want)


@pytest.mark.parametrize("ldd_pad,lead", [(0, 0), (8, 0), (3, 0), (8, 1)])
def test_fused_bf16_guard_bands(ldd_pad, lead):
    """A bf16 D with row padding and odd offsets: nothing outside M x N is
    written (TMA path when 16-byte aligned, plain stores otherwise)."""
    M, N, K = 150, 200, 96
    ldd = N + ldd_pad
    A, B = synth.make_int_inputs(1, M, N, K, seed=ldd_pad + 1)
    sentinel = -1024.0  # exact in bf16
    buf = torch.full((lead + (M + 2) * ldd,), sentinel, dtype=torch.bfloat16, device=dev())
    D = buf[lead: lead + M * ldd].view(M, ldd)[:, :N]
    tg.gemm_fused(A.to(dev()), B.to(dev()), D)
    assert tg.device_error() == tg.TG_OK
    host = buf.float().cpu().numpy()
    mask = np.zeros(host.shape, dtype=bool)
    for i in range(M):
        mask[lead + i * ldd: lead + i * ldd + N] = True
    assert np.all(host[~mask] == sentinel)
    want = _to_bf16(oracle.gemm_dense_f64(A, B).astype(np.float32))
    assert torch.equal(D.cpu().view(torch.int16), want.view(torch.int16))


def test_fused_in_place_residual():
    """R may be D itself: D = A B + D."""
    M, N, K = 200, 256, 300
    A, B = synth.make_int_inputs(1, M, N, K, seed=4)
    D0 = torch.randint(-50, 50, (M, N)).float()
    D = D0.to(dev())
    tg.gemm_fused(A.to(dev()), B.to(dev()), D, residual=D, beta=1.0)
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(D.cpu().numpy(), oracle.gemm_dense_f64(A, B) + D0.numpy())


def test_fused_invalid_arguments():
    A = torch.zeros(8, 8, dtype=torch.bfloat16, device=dev())
    B = torch.zeros(8, 8, dtype=torch.bfloat16, device=dev())
    D = torch.zeros(8, 8, dtype=torch.float32, device=dev())
    e = tg.tg_epilogue()
    e.alpha = 1.0
    e.activation = 7
    assert tg.tg_gemm_fused(A.data_ptr(), B.data_ptr(), D.data_ptr(), 8, 8, 8, 8, 8, 8, 1, 64, 64, 64, e) \
        == tg.TG_ERR_INVALID_ARG
    e.activation = 0
    e.out_type = 5
    assert tg.tg_gemm_fused(A.data_ptr(), B.data_ptr(), D.data_ptr(), 8, 8, 8, 8, 8, 8, 1, 64, 64, 64, e) \
        == tg.TG_ERR_INVALID_ARG
    e.out_type = 0
    R = torch.zeros(8, 16, dtype=torch.float32, device=dev())
    e.residual = R.data_ptr() + 4 * 4  # overlaps nothing of D, but ldr < N
    e.ldr = 4
    assert tg.tg_gemm_fused(A.data_ptr(), B.data_ptr(), D.data_ptr(), 8, 8, 8, 8, 8, 8, 1, 64, 64, 64, e) \
        == tg.TG_ERR_INVALID_ARG
    e.residual = D.data_ptr() + 4  # partial overlap with D
    e.ldr = 8
    assert tg.tg_gemm_fused(A.data_ptr(), B.data_ptr(), D.data_ptr(), 8, 8, 8, 8, 8, 8, 1, 64, 64, 64, e) \
        == tg.TG_ERR_INVALID_ARG
