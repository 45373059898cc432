"""GPU parity of the 8-bit floating-point GEMM (tg_gemm_fp8) against the
fp64 oracle of ``oracle.fp8``, through the C ABI.

Integer-valued inputs (|x| <= 16 in E4M3, <= 8 in E5M2) make every product
and partial sum an exact fp32 integer, so the GPU must equal the oracle bit
for bit; other inputs use the bf16 path's tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import assert_close, dev
from oracle import fp8 as ofp8

pytestmark = pytest.mark.gpu

CONFIGS = [(128, 1), (192, 1), (256, 1), (256, 2)]  # (block_n, cta_pair) with 8-bit instances


def _run(Ac, Btc, fa, fb, options=None, out_dtype=None, **ep):
    A = Ac.to(dev()).view(synth.FP8_DTYPES[fa])
    Bt = Btc.to(dev()).view(synth.FP8_DTYPES[fb])
    D = tg.gemm_fp8(A, Bt, options=options, out_dtype=out_dtype, **ep)
    assert tg.device_error() == tg.TG_OK
    return D.cpu().double().numpy()


def _cfg_id(c):
    return f"bn{c[0]}{'-pair' if c[1] == 2 else ''}"


@pytest.mark.parametrize("cfg", CONFIGS, ids=_cfg_id)
@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (7, 5, 16), (129, 255, 272), (200, 300, 48),
                                   (128, 128, 128), (257, 389, 1040), (300, 130, 4096)])
def test_exact_integer_e4m3(cfg, M, N, K):
    bn, pair = cfg
    A = synth.make_fp8_codes((M, K), 0, seed=M + K)
    Bt = synth.make_fp8_codes((N, K), 0, seed=N + 3 * K)
    got = _run(A, Bt, 0, 0, options=tg.make_options(block_n=bn, cta_pair=pair))
    assert np.array_equal(got, ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), 0, 0))


@pytest.mark.parametrize("fa,fb", [(1, 0), (0, 1), (1, 1)])
def test_exact_integer_mixed_formats(fa, fb):
    M, N, K = 190, 333, 528
    A = synth.make_fp8_codes((M, K), fa, seed=11 + fa)
    Bt = synth.make_fp8_codes((N, K), fb, seed=13 + fb)
    got = _run(A, Bt, fa, fb)
    assert np.array_equal(got, ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), fa, fb))


@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 1), (0, 1)])
@pytest.mark.parametrize("kind", ["finite", "normal"])
def test_float_parity(fa, fb, kind):
    M, N, K = 300, 260, 1024
    A = synth.make_fp8_codes((M, K), fa, seed=21, kind=kind)
    Bt = synth.make_fp8_codes((N, K), fb, seed=22, kind=kind)
    assert_close(_run(A, Bt, fa, fb), ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), fa, fb), K, f"{kind} {fa}{fb}")


def test_batched_split_and_stream_k():
    batch, M, N, K = 3, 150, 290, 2048
    A = synth.make_fp8_codes((batch, M, K), 0, seed=5)
    Bt = synth.make_fp8_codes((batch, N, K), 0, seed=6)
    want = ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), 0, 0)
    for opts in ({}, {"split_k": 3, "cta_pair": 1}, {"stream_k": 2, "block_n": 256, "cta_pair": 2}):
        got = _run(A, Bt, 0, 0, options=tg.make_options(**opts))
        assert np.array_equal(got, want), opts


@pytest.mark.parametrize("bn,pair,depths", [(128, 1, [2, 4, 6]), (192, 1, [2, 4]), (256, 1, [2, 4]),
                                            (256, 2, [2, 4, 6])])
def test_ring_depth_bitwise_invariance(bn, pair, depths):
    M, N, K = 300, 520, 1100 // 16 * 16
    A = synth.make_fp8_codes((M, K), 0, seed=9, kind="normal")
    Bt = synth.make_fp8_codes((N, K), 0, seed=10, kind="normal")
    outs = [_run(A, Bt, 0, 0, options=tg.make_options(block_n=bn, cta_pair=pair, stages=s)) for s in depths]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_fused_scale_bias_activation_bf16_out():
    """Per-tensor scales in alpha, a bias and relu, bf16 output: the same
    formula in fp32 on the fp32 product, rounded to bf16 once."""
    M, N, K = 257, 300, 512
    A = synth.make_fp8_codes((M, K), 0, seed=31)
    Bt = synth.make_fp8_codes((N, K), 0, seed=32)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3))
    scale = 0.0625  # exact: the fused result equals the formula on the exact product
    got = _run(A, Bt, 0, 0, out_dtype=torch.bfloat16, scale=scale, bias=bias.to(dev()), activation="relu")
    C = ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), 0, 0).astype(np.float32)
    x = np.maximum(np.float32(scale) * C + bias.numpy().astype(np.float32)[None, :], np.float32(0))
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)


def test_layout_requirements():
    """Rows not a multiple of 16 bytes are refused (no pack for 8-bit
    operands); a transposed-layout option is an argument error."""
    M, N, K = 64, 64, 40
    A = torch.zeros(M, K, dtype=torch.uint8, device=dev())
    Bt = torch.zeros(N, 48, dtype=torch.uint8, device=dev())
    D = torch.empty(M, N, device=dev())
    st = tg.tg_gemm_fp8(A.data_ptr(), Bt.data_ptr(), D.data_ptr(), M, N, K, K, 48, N, 1, 0, 0, 0, 0, 0)
    assert st == tg.TG_ERR_UNSUPPORTED
    st = tg.tg_gemm_fp8(Bt.data_ptr(), Bt.data_ptr(), D.data_ptr(), M, N, 48, 48, 48, N, 1, 0, 0, 0, 0, 0,
                        None, None, tg.make_options(a_col_major=1))
    assert st == tg.TG_ERR_INVALID_ARG
    st = tg.tg_gemm_fp8(Bt.data_ptr(), Bt.data_ptr(), D.data_ptr(), M, N, 48, 48, 48, N, 1, 0, 0, 0, 2, 0)
    assert st == tg.TG_ERR_INVALID_ARG
