"""GPU parity of the block-scaled 4-bit GEMM (tg_gemm_mxfp4, MXFP4: packed
E2M1 elements, E8M0 scales per 32 elements of K) against the fp64 oracle of
``oracle.mx``, through the C ABI.

Every E2M1 value is a multiple of 1/2 with magnitude at most 6; with scales
2^-1 .. 2^1 every scaled product is a multiple of 1/16 of magnitude at most
144, so for K <= 4096 every partial sum is exact in fp32 and the GPU must
equal the oracle bit for bit whatever its summation order.  Per-row and
per-column power-of-two scales over a wide exponent range are exact too (the
sum is a multiple of one power of two).  Random scales use the bf16 path's
tolerance."""
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


def _inputs(lead, M, N, K, seed, slo=126, shi=128):
    Ac = synth.make_fp4_codes(lead + (M, K), seed=seed)
    Bc = synth.make_fp4_codes(lead + (N, K), seed=seed + 1)
    sfa = synth.make_e8m0_codes(lead + (M, _runs(K)), seed=seed + 2, lo=slo, hi=shi)
    sfb = synth.make_e8m0_codes(lead + (N, _runs(K)), seed=seed + 3, lo=slo, hi=shi)
    return Ac, Bc, sfa, sfb


def _run(Ac, Bc, sfa, sfb, options=None, out_dtype=None, **ep):
    A = synth.pack_fp4_codes(Ac).to(dev())
    Bt = synth.pack_fp4_codes(Bc).to(dev())
    D = tg.gemm_mxfp4(A, Bt, sfa.to(dev()), sfb.to(dev()), options=options, out_dtype=out_dtype, **ep)
    assert tg.device_error() == tg.TG_OK
    return D.cpu().double().numpy()


def _oracle(Ac, Bc, sfa, sfb):
    K = Ac.shape[-1]
    return omx.gemm_mxfp4_f64(omx.pack_fp4(Ac.numpy()), omx.pack_fp4(Bc.numpy()), K, sfa.numpy(), sfb.numpy())


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (7, 5, 96), (128, 128, 256), (129, 255, 544),
                                   (200, 300, 160), (257, 389, 1056), (300, 130, 4096)])
def test_exact_integer(M, N, K):
    Ac, Bc, sfa, sfb = _inputs((), M, N, K, seed=M + 3 * K)
    got = _run(Ac, Bc, sfa, sfb)
    assert np.array_equal(got, _oracle(Ac, Bc, sfa, sfb))


@pytest.mark.parametrize("bn", [128, 192, 224])
@pytest.mark.parametrize("M,N,K", [(130, 224, 512), (129, 225, 160), (257, 447, 800), (64, 465, 2048)])
def test_exact_integer_tile_widths(bn, M, N, K):
    """Every 4-bit tile width; N around the 192- and 224-column tiles and the
    128-column scale blocks inside them; K tails inside a 256-element
    k-block, in both of its scale halves."""
    Ac, Bc, sfa, sfb = _inputs((), M, N, K, seed=M + 5 * K + bn)
    got = _run(Ac, Bc, sfa, sfb, options=tg.make_options(block_n=bn))
    assert np.array_equal(got, _oracle(Ac, Bc, sfa, sfb)), bn


def test_tile_widths_and_rings_bitwise_equal():
    Ac, Bc, sfa, sfb = _inputs((), 300, 500, 1280, seed=17)
    outs = [_run(Ac, Bc, sfa, sfb, options=tg.make_options(block_n=bn, stages=st))
            for bn, st in ((128, 2), (128, 4), (192, 2), (192, 4), (224, 2))]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_k_not_a_multiple_of_32_with_padded_rows():
    """K = 70: the last scale block covers 6 elements, the rows are stored
    with a 96-element pitch (16-byte rows) and the padding is never read."""
    M, N, K, pitch = 90, 150, 70, 96
    Ac, Bc, sfa, sfb = _inputs((), M, N, K, seed=23)
    pad_a = torch.cat([Ac, torch.full((M, pitch - K), 7, dtype=torch.uint8)], dim=1)  # 7: value 6
    pad_b = torch.cat([Bc, torch.full((N, pitch - K), 7, dtype=torch.uint8)], dim=1)
    A = synth.pack_fp4_codes(pad_a).to(dev())[:, : K // 2]
    Bt = synth.pack_fp4_codes(pad_b).to(dev())[:, : K // 2]
    D = tg.gemm_mxfp4(A, Bt, sfa.to(dev()), sfb.to(dev()))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(D.cpu().double().numpy(), _oracle(Ac, Bc, sfa, sfb))


def test_unit_scales_equal_the_8bit_path():
    """With every scale 2^0, MXFP4 equals tg_gemm_fp8 on the same values as
    E4M3 codes (every E2M1 value is an E4M3 value) bit for bit."""
    M, N, K = 200, 330, 1024
    Ac, Bc, _, _ = _inputs((), M, N, K, seed=29)
    one_a = torch.full((M, _runs(K)), 127, dtype=torch.uint8)
    one_b = torch.full((N, _runs(K)), 127, dtype=torch.uint8)
    got = _run(Ac, Bc, one_a, one_b)
    e4m3 = ofp8.table(0)
    lut = np.array([int(np.flatnonzero(e4m3 == v)[0]) if v != 0 else (0x80 if np.signbit(v) else 0)
                    for v in omx.e2m1_table()], dtype=np.uint8)
    A8 = torch.from_numpy(lut[Ac.numpy()]).to(dev()).view(torch.float8_e4m3fn)
    B8 = torch.from_numpy(lut[Bc.numpy()]).to(dev()).view(torch.float8_e4m3fn)
    ref = tg.gemm_fp8(A8, B8).cpu().double().numpy()
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(got, ref)


def test_wide_exponent_range_row_and_column_scales():
    """One scale per row of A and per column of B (the same code in all of a
    row's blocks) over 2^-30 .. 2^30: every output is an exact fp32 value."""
    M, N, K = 150, 260, 512
    Ac, Bc, _, _ = _inputs((), M, N, K, seed=31)
    ra = synth.make_e8m0_codes((M, 1), seed=32, lo=97, hi=157)
    rb = synth.make_e8m0_codes((N, 1), seed=33, lo=97, hi=157)
    sfa = ra.repeat(1, _runs(K)).contiguous()
    sfb = rb.repeat(1, _runs(K)).contiguous()
    assert np.array_equal(_run(Ac, Bc, sfa, sfb), _oracle(Ac, Bc, sfa, sfb))


def test_float_parity_random_scales():
    M, N, K = 333, 777, 2048
    Ac, Bc, sfa, sfb = _inputs((), M, N, K, seed=37, slo=110, shi=140)
    assert_close(_run(Ac, Bc, sfa, sfb), _oracle(Ac, Bc, sfa, sfb), K, "mxfp4 random scales")


def test_batched_split_and_stream_k():
    lead = (3,)
    Ac, Bc, sfa, sfb = _inputs(lead, 140, 270, 1536, seed=41)
    ref = _oracle(Ac, Bc, sfa, sfb)
    assert np.array_equal(_run(Ac, Bc, sfa, sfb), ref)
    assert np.array_equal(_run(Ac, Bc, sfa, sfb, options=tg.make_options(split_k=3)), ref)
    assert np.array_equal(_run(Ac, Bc, sfa, sfb, options=tg.make_options(block_n=128, max_ctas=5, stream_k=2)),
                          ref)


def test_shared_operand_and_scales():
    """B and its scales shared by every problem of the batch (stride 0)."""
    Ac, _, sfa, _ = _inputs((4,), 100, 1, 640, seed=43)
    _, Bc, _, sfb = _inputs((), 1, 200, 640, seed=44)
    A = synth.pack_fp4_codes(Ac).to(dev())
    Bt = synth.pack_fp4_codes(Bc).to(dev()).unsqueeze(0).expand(4, -1, -1)
    sfb_d = sfb.to(dev()).unsqueeze(0).expand(4, -1, -1)
    D = tg.gemm_mxfp4(A, Bt, sfa.to(dev()), sfb_d)
    assert tg.device_error() == tg.TG_OK
    ref = omx.gemm_mxfp4_f64(omx.pack_fp4(Ac.numpy()), omx.pack_fp4(Bc.numpy())[None], 640, sfa.numpy(),
                             sfb.numpy()[None])
    assert np.array_equal(D.cpu().double().numpy(), ref)


def test_fused_scale_bias_activation_bf16_out():
    M, N, K = 130, 200, 768
    Ac, Bc, sfa, sfb = _inputs((), M, N, K, seed=47)
    bias = torch.linspace(-3, 3, N, dtype=torch.float32)
    got = _run(Ac, Bc, sfa, sfb, out_dtype=torch.bfloat16, scale=0.25, bias=bias.to(dev()), activation="relu")
    raw = _oracle(Ac, Bc, sfa, sfb)
    ref = np.maximum(np.float32(0.25) * raw.astype(np.float32) + bias.numpy(), 0)
    want = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)


def test_argument_errors():
    # 64-byte rows allocated, so that pitches up to 128 elements stay inside
    A = torch.zeros(64, 64, dtype=torch.uint8, device=dev())
    Bt = torch.zeros(64, 64, dtype=torch.uint8, device=dev())
    D = torch.zeros(64, 64, dtype=torch.float32, device=dev())
    sf = torch.zeros(64, 2, dtype=torch.uint8, device=dev())
    s = torch.cuda.current_stream().cuda_stream

    def call(K=64, lda=64, ldb=64, opt=None):
        return tg.tg_gemm_mxfp4(A.data_ptr(), Bt.data_ptr(), D.data_ptr(), 64, 64, K, lda, ldb, 64, 1, 0, 0, 0,
                                sf.data_ptr(), 2, 0, sf.data_ptr(), 2, 0, None, s, opt)
    assert call(K=63, lda=64) == tg.TG_ERR_INVALID_ARG        # K odd: half a byte
    assert call(lda=65) == tg.TG_ERR_INVALID_ARG              # odd pitch
    assert call(lda=80, ldb=80) == tg.TG_ERR_UNSUPPORTED       # 40-byte rows: not 16-byte aligned
    assert call(opt=tg.make_options(block_n=224, stages=4)) == tg.TG_ERR_INVALID_ARG
    assert call(opt=tg.make_options(block_n=256)) == tg.TG_ERR_INVALID_ARG
    assert call() == tg.TG_OK
    assert tg.device_error() == tg.TG_OK
