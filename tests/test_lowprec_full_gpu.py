"""Full-size parity of the 8-bit and 4-bit entry points in the launch
configurations ``bench.py --dtype e4m3 / mxfp8 / mxfp4`` times (4096^3,
default plans), and of the 8-bit skinny shape 64 x 28672 x 8192 (its
64-row A rings): EVERY element of the output against the fp64 oracle.

Inputs are exact: E4M3 integers in [-16, 16] (products up to 256, sums up
to 256 K < 2^24 - exact in fp32), MXFP8 the same with E8M0 scales 2^-1 ..
2^1, MXFP4 E2M1 codes with the same scales (every partial sum a multiple of
1/16 far below 2^20), so the GPU must equal the oracle bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev
from oracle import fp8 as ofp8
from oracle import mx as omx

pytestmark = pytest.mark.gpu


def _runs(K):
    return -(-K // 32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tg.load()
    yield


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (64, 28672, 8192)])
def test_e4m3_full_output(M, N, K):
    A = synth.make_fp8_codes((M, K), 0, seed=M + 7)
    Bt = synth.make_fp8_codes((N, K), 0, seed=N + 11)
    D = tg.gemm_fp8(A.to(dev()).view(torch.float8_e4m3fn), Bt.to(dev()).view(torch.float8_e4m3fn))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(D.cpu().double().numpy(), ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), 0, 0))


def test_mxfp8_full_output():
    M = N = K = 4096
    A = synth.make_fp8_codes((M, K), 0, seed=21)
    Bt = synth.make_fp8_codes((N, K), 0, seed=22)
    sfa = synth.make_e8m0_codes((M, _runs(K)), seed=23, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, _runs(K)), seed=24, lo=126, hi=128)
    D = tg.gemm_mxfp8(A.to(dev()).view(torch.float8_e4m3fn), Bt.to(dev()).view(torch.float8_e4m3fn),
                      sfa.to(dev()), sfb.to(dev()))
    assert tg.device_error() == tg.TG_OK
    ref = omx.gemm_mx_f64(A.numpy(), Bt.numpy(), 0, 0, sfa.numpy(), sfb.numpy())
    assert np.array_equal(D.cpu().double().numpy(), ref)


def test_mxfp4_full_output():
    M = N = K = 4096
    Ac = synth.make_fp4_codes((M, K), seed=31)
    Bc = synth.make_fp4_codes((N, K), seed=32)
    sfa = synth.make_e8m0_codes((M, _runs(K)), seed=33, lo=126, hi=128)
    sfb = synth.make_e8m0_codes((N, _runs(K)), seed=34, lo=126, hi=128)
    D = tg.gemm_mxfp4(synth.pack_fp4_codes(Ac).to(dev()), synth.pack_fp4_codes(Bc).to(dev()), sfa.to(dev()),
                      sfb.to(dev()))
    assert tg.device_error() == tg.TG_OK
    ref = omx.gemm_mxfp4_f64(omx.pack_fp4(Ac.numpy()), omx.pack_fp4(Bc.numpy()), K, sfa.numpy(), sfb.numpy())
    assert np.array_equal(D.cpu().double().numpy(), ref)
