"""GPU parity of the block-scaled 8-bit GEMM (tg_gemm_mxfp8) against the
fp64 oracle of ``oracle.mx``, through the C ABI.

Integer-valued elements with scales 2^-1 .. 2^1 keep every scaled product a
multiple of 1/4 and every partial sum far below 2^22, so the GPU must equal
the oracle bit for bit; per-row / per-column power-of-two scales over a wide
exponent range are exact too (the sum is an integer times one power of
two).  Random-valued elements use the bf16 path's tolerance."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import assert_close, dev
from oracle import fp8 as ofp8
from oracle import mx as omx

pytestmark = pytest.mark.gpu


def _runs(K):
    return -(-K // 32)


def _run(Ac, Btc, sfa, sfb, fa=0, fb=0, options=None, out_dtype=None, **ep):
    A = Ac.to(dev()).view(synth.FP8_DTYPES[fa])
    Bt = Btc.to(dev()).view(synth.FP8_DTYPES[fb])
    D = tg.gemm_mxfp8(A, Bt, sfa.to(dev()), sfb.to(dev()), options=options, out_dtype=out_dtype, **ep)
    assert tg.device_error() == tg.TG_OK
    return D.cpu().double().numpy()


def _oracle(A, Bt, sfa, sfb, fa=0, fb=0):
    return omx.gemm_mx_f64(A.numpy(), Bt.numpy(), fa, fb, sfa.numpy(), sfb.numpy())


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (7, 5, 48), (129, 255, 272), (128, 128, 128),
                                   (200, 300, 80), (257, 389, 1040), (300, 130, 4096)])
def test_exact_integer(M, N, K):
    A = synth.make_fp8_codes((M, K), 0, seed=M + K)
    Bt = synth.make_fp8_codes((N, K), 0, seed=N + 3 * K)
    sfa = synth.make_e8m0_codes((M, _runs(K)), seed=1 + M, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, _runs(K)), seed=2 + N, lo=126, hi=128)
    got = _run(A, Bt, sfa, sfb)
    assert np.array_equal(got, _oracle(A, Bt, sfa, sfb))


@pytest.mark.parametrize("bn", [128, 192, 224])
@pytest.mark.parametrize("M,N,K", [(130, 224, 256), (129, 225, 160), (257, 447, 528), (64, 465, 1024),
                                   (300, 700, 2080)])
def test_exact_integer_tile_widths(bn, M, N, K):
    """Every block-scaled tile width; N around the 192- and 224-column tiles
    and the 128-column scale blocks inside them."""
    A = synth.make_fp8_codes((M, K), 0, seed=M + 5 * K)
    Bt = synth.make_fp8_codes((N, K), 0, seed=N + 7 * K)
    sfa = synth.make_e8m0_codes((M, _runs(K)), seed=3 + M, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, _runs(K)), seed=4 + N, lo=126, hi=128)
    got = _run(A, Bt, sfa, sfb, options=tg.make_options(block_n=bn))
    assert np.array_equal(got, _oracle(A, Bt, sfa, sfb))


def test_tile_widths_bitwise_equal():
    """Each output element sees the same MMA sequence at either width."""
    M, N, K = 300, 520, 1024
    A = synth.make_fp8_codes((M, K), 0, seed=61, kind="normal")
    Bt = synth.make_fp8_codes((N, K), 0, seed=62, kind="normal")
    sfa = synth.make_e8m0_codes((M, K // 32), seed=63)
    sfb = synth.make_e8m0_codes((N, K // 32), seed=64)
    outs = [_run(A, Bt, sfa, sfb, options=tg.make_options(block_n=bn, stream_k=1)) for bn in (128, 192, 224)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert_close(outs[2], _oracle(A, Bt, sfa, sfb), K, "224 vs oracle")


@pytest.mark.parametrize("fa,fb", [(1, 0), (0, 1), (1, 1)])
def test_exact_integer_mixed_formats(fa, fb):
    M, N, K = 190, 333, 528
    A = synth.make_fp8_codes((M, K), fa, seed=11 + fa)
    Bt = synth.make_fp8_codes((N, K), fb, seed=13 + fb)
    sfa = synth.make_e8m0_codes((M, _runs(K)), seed=5, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, _runs(K)), seed=6, lo=126, hi=128)
    got = _run(A, Bt, sfa, sfb, fa, fb)
    assert np.array_equal(got, _oracle(A, Bt, sfa, sfb, fa, fb))


def test_unit_scales_equal_unscaled_fp8():
    """Scale code 127 (2^0) everywhere: the unscaled 8-bit GEMM, bit for bit."""
    M, N, K = 300, 260, 1024
    A = synth.make_fp8_codes((M, K), 0, seed=21, kind="normal")
    Bt = synth.make_fp8_codes((N, K), 0, seed=22, kind="normal")
    ones_a = torch.full((M, K // 32), 127, dtype=torch.uint8)
    ones_b = torch.full((N, K // 32), 127, dtype=torch.uint8)
    got = _run(A, Bt, ones_a, ones_b)
    plain = tg.gemm_fp8(A.to(dev()).view(torch.float8_e4m3fn), Bt.to(dev()).view(torch.float8_e4m3fn))
    assert np.array_equal(got, plain.cpu().double().numpy())
    assert_close(got, ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), 0, 0), K, "unit scales")


def test_wide_exponent_range_row_and_column_scales():
    """One scale per row of A and per column of B (the same code for all of
    a row's runs), codes 97 .. 157: C[i][j] = 2^(a_i + b_j) * (integer sum),
    exact in fp32."""
    M, N, K = 256, 384, 640
    A = synth.make_fp8_codes((M, K), 0, seed=41)
    Bt = synth.make_fp8_codes((N, K), 0, seed=42)
    ra = synth.make_e8m0_codes((M, 1), seed=43, lo=97, hi=157)
    rb = synth.make_e8m0_codes((N, 1), seed=44, lo=97, hi=157)
    sfa = ra.expand(M, _runs(K)).contiguous()
    sfb = rb.expand(N, _runs(K)).contiguous()
    got = _run(A, Bt, sfa, sfb)
    assert np.array_equal(got, _oracle(A, Bt, sfa, sfb))


@pytest.mark.parametrize("fa,fb", [(0, 0), (1, 1), (0, 1)])
@pytest.mark.parametrize("kind", ["finite", "normal"])
def test_float_parity(fa, fb, kind):
    M, N, K = 300, 260, 1024
    A = synth.make_fp8_codes((M, K), fa, seed=21, kind=kind)
    Bt = synth.make_fp8_codes((N, K), fb, seed=22, kind=kind)
    sfa = synth.make_e8m0_codes((M, K // 32), seed=23)
    sfb = synth.make_e8m0_codes((N, K // 32), seed=24)
    assert_close(_run(A, Bt, sfa, sfb, fa, fb), _oracle(A, Bt, sfa, sfb, fa, fb), K, f"{kind} {fa}{fb}")


def test_batched_split_and_stream_k():
    batch, M, N, K = 3, 150, 290, 2048
    A = synth.make_fp8_codes((batch, M, K), 0, seed=5)
    Bt = synth.make_fp8_codes((batch, N, K), 0, seed=6)
    sfa = synth.make_e8m0_codes((batch, M, K // 32), seed=7, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((batch, N, K // 32), seed=8, lo=126, hi=128)
    want = _oracle(A, Bt, sfa, sfb)
    for opts in ({}, {"split_k": 3}, {"stream_k": 2}, {"stages": 2}):
        got = _run(A, Bt, sfa, sfb, options=tg.make_options(**opts))
        assert np.array_equal(got, want), opts


def test_shared_operand_and_scales():
    """A shared across the batch (stride 0) with shared scales; B's scales
    shared while B is not."""
    batch, M, N, K = 2, 140, 200, 512
    A = synth.make_fp8_codes((M, K), 0, seed=51)
    Bt = synth.make_fp8_codes((batch, N, K), 0, seed=52)
    sfa = synth.make_e8m0_codes((M, K // 32), seed=53, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, K // 32), seed=54, lo=126, hi=128)
    got = _run(A, Bt, sfa, sfb)
    want = np.stack([_oracle(A, Bt[b], sfa, sfb) for b in range(batch)])
    assert np.array_equal(got, want)


@pytest.mark.parametrize("bn", [128, 192, 224])
def test_ring_depth_bitwise_invariance(bn):
    M, N, K = 300, 520, 1088
    A = synth.make_fp8_codes((M, K), 0, seed=9, kind="normal")
    Bt = synth.make_fp8_codes((N, K), 0, seed=10, kind="normal")
    sfa = synth.make_e8m0_codes((M, _runs(K)), seed=11)
    sfb = synth.make_e8m0_codes((N, _runs(K)), seed=12)
    outs = [_run(A, Bt, sfa, sfb, options=tg.make_options(stages=s, block_n=bn)) for s in (2, 4)]
    assert np.array_equal(outs[0], outs[1])


def test_fused_scale_bias_activation_bf16_out():
    M, N, K = 257, 300, 512
    A = synth.make_fp8_codes((M, K), 0, seed=31)
    Bt = synth.make_fp8_codes((N, K), 0, seed=32)
    sfa = synth.make_e8m0_codes((M, K // 32), seed=33, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, K // 32), seed=34, lo=126, hi=128)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3))
    scale = 0.0625
    got = _run(A, Bt, sfa, sfb, out_dtype=torch.bfloat16, scale=scale, bias=bias.to(dev()), activation="relu")
    C = _oracle(A, Bt, sfa, sfb).astype(np.float32)
    x = np.maximum(np.float32(scale) * C + bias.numpy().astype(np.float32)[None, :], np.float32(0))
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)


def test_argument_errors():
    M, N, K = 64, 64, 64
    A = torch.zeros(M, K, dtype=torch.uint8, device=dev())
    Bt = torch.zeros(N, K, dtype=torch.uint8, device=dev())
    D = torch.empty(M, N, device=dev())
    sf = torch.full((max(M, N), 2), 127, dtype=torch.uint8, device=dev())
    p = sf.data_ptr()

    def call(sfa=p, ld_sfa=2, sfb=p, ld_sfb=2, opt=None, batch=1, sA=0, s_sfa=0):
        return tg.tg_gemm_mxfp8(A.data_ptr(), Bt.data_ptr(), D.data_ptr(), M, N, K, K, K, N, batch, sA, 0,
                                M * N, 0, 0, sfa, ld_sfa, s_sfa, sfb, ld_sfb, 0, None, None, opt)

    assert call() == tg.TG_OK
    assert call(sfa=None) == tg.TG_ERR_INVALID_ARG
    assert call(ld_sfb=1) == tg.TG_ERR_INVALID_ARG
    assert call(opt=tg.make_options(block_n=256)) == tg.TG_ERR_INVALID_ARG
    assert call(opt=tg.make_options(block_n=224)) == tg.TG_OK
    assert call(opt=tg.make_options(block_n=192)) == tg.TG_OK
    assert call(opt=tg.make_options(block_n=64)) == tg.TG_ERR_INVALID_ARG
    assert call(opt=tg.make_options(cta_pair=2)) == tg.TG_ERR_INVALID_ARG
    assert call(opt=tg.make_options(stages=6)) == tg.TG_ERR_INVALID_ARG
    assert call(s_sfa=-1) == tg.TG_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert tg.device_error() == tg.TG_OK


@pytest.mark.parametrize("bn", [128, 192, 224])
def test_scale_pitches_agree(bn):
    """The same scales at two pitches (a multiple of 4 and an odd one),
    batched, with a K whose last run is partial: bit for bit equal, and equal
    to the oracle."""
    batch, M, N, K = 2, 260, 470, 1040
    runs = K // 32 + 1  # 33 runs, the last one half full
    A = synth.make_fp8_codes((batch, M, K), 0, seed=71)
    Bt = synth.make_fp8_codes((batch, N, K), 0, seed=72)
    sfa = synth.make_e8m0_codes((batch, M, runs), seed=73, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((batch, N, runs), seed=74, lo=126, hi=128)
    want = _oracle(A, Bt, sfa, sfb)
    outs = []
    for pitch in (36, 35):
        fa = torch.full((batch, M, pitch), 255, dtype=torch.uint8)
        fa[:, :, :runs] = sfa
        fb = torch.full((batch, N, pitch), 255, dtype=torch.uint8)
        fb[:, :, :runs] = sfb
        Ad = A.to(dev()).view(torch.float8_e4m3fn)
        Bd = Bt.to(dev()).view(torch.float8_e4m3fn)
        D = tg.gemm_mxfp8(Ad, Bd, fa.to(dev())[:, :, :runs], fb.to(dev())[:, :, :runs],
                          options=tg.make_options(block_n=bn))
        assert tg.device_error() == tg.TG_OK
        outs.append(D.cpu().double().numpy())
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(outs[0], want)
