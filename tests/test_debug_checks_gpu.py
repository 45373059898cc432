"""The TG_DEBUG_CHECKS build of the library beside the product build.

That build verifies on the device, before each access, its work units, ring
slots, tensor-memory columns, shared-memory layout and split-K scratch
indices (the checks the sanitizer would otherwise stand in for; it is not
available here).  Run over plans that exercise every path - tile widths,
two-SM tiles, split-K, stream-K, batched, transposed operands, the fused
epilogue, 8-bit and block-scaled operands - it must report no failed check
and produce bit-for-bit the product build's output.  A planted failure
(debug_stall = 2) must come back as TG_ERR_DEVICE_CHECK, after which the
next call is exact again.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev, oracle_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    return tg.load(), tg.load_checks()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _gemm(lib, A, B, C, opt):
    batch = A.shape[0] if A.dim() == 3 else 1
    M, K = A.shape[-2:]
    N = B.shape[-1]
    st = lib.tg_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, A.stride(-2), B.stride(-2),
                        C.stride(-2), batch, M * A.stride(-2) if batch > 1 else 0,
                        K * B.stride(-2) if batch > 1 else 0, M * C.stride(-2) if batch > 1 else 0, _stream(),
                        ctypes.byref(opt) if opt is not None else None)
    return st


CASES = [
    ("default ragged", (1, 197, 131, 77), {}),
    ("width 64", (1, 300, 300, 500), dict(block_n=64)),
    ("width 192", (1, 257, 385, 300), dict(block_n=192, cta_pair=1)),
    ("pair 256", (1, 520, 600, 700), dict(block_n=256, cta_pair=2)),
    ("pair 128 ring 8", (1, 513, 260, 640), dict(block_n=128, cta_pair=2, stages=8)),
    ("split-K 3", (1, 130, 250, 2000), dict(split_k=3)),
    ("stream-K 7 CTAs", (1, 1000, 1000, 1024), dict(block_n=128, max_ctas=7, stream_k=2)),
    ("stream-K pairs", (1, 1100, 1200, 900), dict(block_n=256, cta_pair=2, max_ctas=10, stream_k=2)),
    ("batched", (5, 150, 170, 333), {}),
    ("one CTA walks all", (1, 400, 400, 256), dict(block_n=128, max_ctas=1)),
]


@pytest.mark.parametrize("name,shape,opts", CASES, ids=[c[0] for c in CASES])
def test_checks_build_agrees_and_reports_nothing(libs, name, shape, opts):
    lib, chk = libs
    batch, M, N, K = shape
    Ai, Bi = synth.make_int_inputs(batch, M, N, K, seed=M + N + K)
    A, B = Ai.to(dev()), Bi.to(dev())
    lead = (batch,) if batch > 1 else ()
    C1 = torch.full(lead + (M, N), float("nan"), device=dev())
    C2 = torch.full(lead + (M, N), float("nan"), device=dev())
    opt = tg.make_options(**opts) if opts else None
    assert _gemm(lib, A, B, C1, opt) == tg.TG_OK
    assert _gemm(chk, A, B, C2, opt) == tg.TG_OK
    assert lib.tg_device_error(_stream()) == tg.TG_OK
    assert chk.tg_device_error(_stream()) == tg.TG_OK, name
    assert torch.equal(C1, C2), name
    assert np.array_equal(C2.cpu().double().numpy(), oracle_dense(Ai, Bi)), name


def test_checks_build_transposed_and_fused(libs):
    lib, chk = libs
    M, N, K = 300, 280, 520
    Ai, Bi = synth.make_int_inputs(1, M, N, K, seed=5)
    At = Ai.t().contiguous().to(dev())  # A stored K x M
    Bt = Bi.t().contiguous().to(dev())  # B stored N x K
    outs = []
    for L in (lib, chk):
        C = torch.empty(M, N, device=dev())
        opt = tg.make_options(a_col_major=1, b_col_major=1)
        st = L.tg_gemm_ex(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), M, N, K, M, K, N, 1, 0, 0, 0, _stream(),
                          ctypes.byref(opt))
        assert st == tg.TG_OK
        assert L.tg_device_error(_stream()) == tg.TG_OK
        outs.append(C)
    assert torch.equal(outs[0], outs[1])
    A, B = Ai.to(dev()), Bi.to(dev())
    bias = torch.linspace(-2, 2, N, device=dev())
    outs = []
    for L in (lib, chk):
        D = torch.empty(M, N, device=dev(), dtype=torch.bfloat16)
        ep = tg.tg_epilogue()
        ep.alpha, ep.beta, ep.bias, ep.activation, ep.out_type = 0.5, 0.0, bias.data_ptr(), tg.TG_ACT_RELU, 1
        st = L.tg_gemm_fused(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, K, N, N, 1, 0, 0, 0,
                             ctypes.byref(ep), _stream(), None)
        assert st == tg.TG_OK
        assert L.tg_device_error(_stream()) == tg.TG_OK
        outs.append(D)
    assert torch.equal(outs[0], outs[1])


def test_checks_build_block_scaled(libs):
    """MXFP8 and MXFP4 (their scale columns in tensor memory are checked)."""
    lib, chk = libs
    M, N, K = 260, 450, 1024
    A8 = synth.make_fp8_codes((M, K), 0, seed=1).to(dev())
    B8 = synth.make_fp8_codes((N, K), 0, seed=2).to(dev())
    sfa = synth.make_e8m0_codes((M, K // 32), seed=3, lo=126, hi=128).to(dev())
    sfb = synth.make_e8m0_codes((N, K // 32), seed=4, lo=126, hi=128).to(dev())
    A4 = synth.pack_fp4_codes(synth.make_fp4_codes((M, K), seed=5)).to(dev())
    B4 = synth.pack_fp4_codes(synth.make_fp4_codes((N, K), seed=6)).to(dev())
    for bn in (128, 192, 224):
        opt = tg.make_options(block_n=bn)
        outs8, outs4 = [], []
        for L in (lib, chk):
            D8 = torch.empty(M, N, device=dev())
            D4 = torch.empty(M, N, device=dev())
            st = L.tg_gemm_mxfp8(A8.data_ptr(), B8.data_ptr(), D8.data_ptr(), M, N, K, K, K, N, 1, 0, 0, 0, 0, 0,
                                 sfa.data_ptr(), K // 32, 0, sfb.data_ptr(), K // 32, 0, None, _stream(),
                                 ctypes.byref(opt))
            assert st == tg.TG_OK
            st = L.tg_gemm_mxfp4(A4.data_ptr(), B4.data_ptr(), D4.data_ptr(), M, N, K, K, K, N, 1, 0, 0, 0,
                                 sfa.data_ptr(), K // 32, 0, sfb.data_ptr(), K // 32, 0, None, _stream(),
                                 ctypes.byref(opt))
            assert st == tg.TG_OK
            assert L.tg_device_error(_stream()) == tg.TG_OK, bn
            outs8.append(D8)
            outs4.append(D4)
        assert torch.equal(outs8[0], outs8[1]), bn
        assert torch.equal(outs4[0], outs4[1]), bn


def test_planted_check_failure_is_reported_and_recovers(libs):
    lib, chk = libs
    M, N, K = 300, 300, 512
    Ai, Bi = synth.make_int_inputs(1, M, N, K, seed=9)
    A, B = Ai.to(dev()), Bi.to(dev())
    C = torch.empty(M, N, device=dev())
    for opts in (dict(block_n=128), dict(block_n=256, cta_pair=2), dict(split_k=2)):
        opt = tg.make_options(debug_stall=2, timeout_ns=20_000_000, **opts)
        assert _gemm(chk, A, B, C, opt) == tg.TG_OK
        assert chk.tg_device_error(_stream()) == tg.TG_ERR_DEVICE_CHECK, opts
        assert chk.tg_device_error(_stream()) == tg.TG_OK
    # in the product build the same option is the watchdog self-test
    opt = tg.make_options(debug_stall=2, timeout_ns=20_000_000, block_n=128)
    assert _gemm(lib, A, B, C, opt) == tg.TG_OK
    assert lib.tg_device_error(_stream()) == tg.TG_ERR_TIMEOUT
    C.fill_(float("nan"))
    assert _gemm(chk, A, B, C, tg.make_options(split_k=2)) == tg.TG_OK
    assert chk.tg_device_error(_stream()) == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(Ai, Bi))
