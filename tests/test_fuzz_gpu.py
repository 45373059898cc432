"""Randomised exact-integer parity of the CUDA path: random extents,
layouts (row- or column-major A and B), operand offsets and pitches,
batch strides and plan overrides, each compared with the fp64 oracle bit
for bit.  The cases are drawn from a fixed seed, so a failure reproduces."""
from __future__ import annotations

import random

import numpy as np
import pytest
import torch

import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import dev, oracle_dense

pytestmark = pytest.mark.gpu

N_CASES = 60


def _case(i):
    r = random.Random(1000 + i)
    M, N, K = r.randint(1, 700), r.randint(1, 700), r.randint(1, 900)
    batch = r.choice([1, 1, 1, 2, 3])
    a_cm, b_cm = r.random() < 0.3, r.random() < 0.3
    opts = {}
    bn = r.choice([0, 64, 128, 192, 256])
    if bn:
        opts["block_n"] = bn
    pair = r.choice([0, 0, 1, 2])
    if pair == 2 and bn not in (0, 128, 256):
        pair = 0
    if pair:
        opts["cta_pair"] = pair
    kb = (K + 63) // 64
    mode = r.choice(["plain", "plain", "split", "stream"])
    if mode == "split" and kb > 1:
        opts["split_k"] = r.randint(2, min(6, kb))
    if mode == "stream":
        opts["stream_k"] = 2
    return dict(M=M, N=N, K=K, batch=batch, a_cm=a_cm, b_cm=b_cm, opts=opts,
                a_pad=r.choice([0, 0, 1, 8, 13]), b_pad=r.choice([0, 0, 3, 8]),
                c_pad=r.choice([0, 0, 5, 4]), a_off=r.choice([0, 0, 1, 4]), seed=r.randint(0, 10 ** 6))


def _place(t, rows, cols, ld, off, stride, batch):
    """Copy [batch, rows, cols] into a zero buffer at element offset `off`
    with row pitch `ld` and problem stride `stride`; return the device
    buffer and the view."""
    buf = torch.zeros(off + (batch - 1) * stride + rows * ld + 8, dtype=t.dtype)
    for b in range(batch):
        buf[off + b * stride: off + b * stride + rows * ld].view(rows, ld)[:, :cols] = t[b]
    d = buf.to(dev())
    return d, torch.as_strided(d, (batch, rows, cols), (stride, ld, 1), off)


def _case_short(i):
    """Outputs of at most 64 rows (the planner's rings of 64-row A slots at
    widths 128 and 192), with long N and K."""
    r = random.Random(9000 + i)
    M, N, K = r.randint(1, 64), r.randint(1, 3000), r.randint(1, 3000)
    opts = {}
    bn = r.choice([0, 128, 128, 192, 192])
    if bn:
        opts["block_n"] = bn
    kb = (K + 63) // 64
    if r.random() < 0.3 and kb > 1:
        opts["split_k"] = r.randint(2, min(8, kb))
    return dict(M=M, N=N, K=K, batch=r.choice([1, 1, 2, 4]), a_cm=r.random() < 0.3, b_cm=r.random() < 0.3,
                opts=opts, a_pad=r.choice([0, 0, 1, 8]), b_pad=r.choice([0, 0, 3, 8]), c_pad=r.choice([0, 0, 5, 4]),
                a_off=r.choice([0, 0, 1, 4]), seed=r.randint(0, 10 ** 6))


def _case_direct(i):
    """The direct-load kernel (direct = 2): operands staged by the threads
    at any pitch, offset and layout, several staged chunks of K."""
    r = random.Random(7000 + i)
    M, N, K = r.randint(1, 400), r.randint(1, 400), r.randint(1, 1200)
    return dict(M=M, N=N, K=K, batch=r.choice([1, 1, 2, 3]), a_cm=r.random() < 0.4, b_cm=r.random() < 0.4,
                opts=dict(direct=2), a_pad=r.choice([0, 1, 8, 13]), b_pad=r.choice([0, 3, 8]),
                c_pad=r.choice([0, 5, 4]), a_off=r.choice([0, 1, 4]), seed=r.randint(0, 10 ** 6))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_exact_cases(i):
    _run_exact_case(_case(i))


@pytest.mark.parametrize("i", range(30))
def test_random_short_outputs(i):
    _run_exact_case(_case_short(i))


@pytest.mark.parametrize("i", range(40))
def test_random_direct_kernel(i):
    _run_exact_case(_case_direct(i))


def _run_exact_case(c):
    M, N, K, batch = c["M"], c["N"], c["K"], c["batch"]
    A, B = synth.make_int_inputs(batch, M, N, K, seed=c["seed"])
    A3 = A.reshape(batch, M, K)
    B3 = B.reshape(batch, K, N)
    # stored layouts: row-major, or the transpose (column-major)
    As = A3.transpose(1, 2).contiguous() if c["a_cm"] else A3
    Bs = B3.transpose(1, 2).contiguous() if c["b_cm"] else B3
    ar, ac = As.shape[1], As.shape[2]
    br, bc = Bs.shape[1], Bs.shape[2]
    lda, ldb, ldc = ac + c["a_pad"], bc + c["b_pad"], N + c["c_pad"]
    sA, sB, sC = ar * lda + 16, br * ldb, M * ldc + 8
    ad, _ = _place(As, ar, ac, lda, c["a_off"], sA, batch)
    bd, _ = _place(Bs, br, bc, ldb, 0, sB, batch)
    cbuf = torch.full(((batch - 1) * sC + M * ldc + 8,), float("nan"), device=dev())
    o = tg.make_options(a_col_major=int(c["a_cm"]), b_col_major=int(c["b_cm"]), **c["opts"])
    st = tg.tg_gemm_ex(ad.data_ptr() + 2 * c["a_off"], bd.data_ptr(), cbuf.data_ptr(), M, N, K, lda, ldb, ldc,
                       batch, sA if batch > 1 else 0, sB if batch > 1 else 0, sC if batch > 1 else 0,
                       torch.cuda.current_stream().cuda_stream, o)
    assert st == tg.TG_OK, (c, tg.STATUS_NAMES.get(st, st))
    assert tg.device_error() == tg.TG_OK, c
    host = cbuf.cpu().numpy()
    want = oracle_dense(A3, B3).reshape(batch, M, N)
    mask = np.zeros(host.shape, dtype=bool)
    for b in range(batch):
        for i_ in range(M):
            lo = b * sC + i_ * ldc
            mask[lo: lo + N] = True
            assert np.array_equal(host[lo: lo + N].astype(np.float64), want[b, i_]), (c, b, i_)
    assert np.all(np.isnan(host[~mask])), ("write outside C", c)


def _case_fp8(i):
    r = random.Random(5000 + i)
    M, N = r.randint(1, 600), r.randint(1, 600)
    K = 16 * r.randint(1, 50)
    batch = r.choice([1, 1, 2])
    cfg = r.choice([(0, 0), (128, 1), (256, 1), (256, 2)])
    opts = {}
    if cfg[0]:
        opts = {"block_n": cfg[0], "cta_pair": cfg[1]}
    if r.random() < 0.25 and K >= 256:
        opts["split_k"] = 2
        opts["cta_pair"] = 1
    return dict(M=M, N=N, K=K, batch=batch, opts=opts, fa=r.choice([0, 1]), fb=r.choice([0, 1]),
                lda_pad=16 * r.choice([0, 0, 1]), ldb_pad=16 * r.choice([0, 1]), ldd_pad=r.choice([0, 3, 8]),
                out=r.choice(["f32", "bf16"]), seed=r.randint(0, 10 ** 6))


@pytest.mark.parametrize("i", range(24))
def test_random_fp8_cases(i):
    """8-bit operands: random extents, pitches, formats, plans and output
    types; exact against the oracle (bf16 output: the exact product rounded
    once), and nothing written outside D."""
    from oracle import fp8 as ofp8

    c = _case_fp8(i)
    M, N, K, batch = c["M"], c["N"], c["K"], c["batch"]
    A = synth.make_fp8_codes((batch, M, K), c["fa"], seed=c["seed"])
    Bt = synth.make_fp8_codes((batch, N, K), c["fb"], seed=c["seed"] + 1)
    lda, ldb, ldd = K + c["lda_pad"], K + c["ldb_pad"], N + c["ldd_pad"]
    abuf = torch.zeros(batch * M * lda, dtype=torch.uint8)
    bbuf = torch.zeros(batch * N * ldb, dtype=torch.uint8)
    abuf.view(batch, M, lda)[:, :, :K] = A
    bbuf.view(batch, N, ldb)[:, :, :K] = Bt
    ad, bd = abuf.to(dev()), bbuf.to(dev())
    dt = torch.float32 if c["out"] == "f32" else torch.bfloat16
    sD = M * ldd + 8
    dbuf = torch.full(((batch - 1) * sD + M * ldd + 8,), float("nan"), dtype=dt, device=dev())
    ep = tg.tg_epilogue()
    ep.alpha, ep.beta = 1.0, 0.0
    ep.out_type = tg.TG_F32 if c["out"] == "f32" else tg.TG_BF16
    st = tg.tg_gemm_fp8(ad.data_ptr(), bd.data_ptr(), dbuf.data_ptr(), M, N, K, lda, ldb, ldd, batch,
                        M * lda if batch > 1 else 0, N * ldb if batch > 1 else 0, sD if batch > 1 else 0,
                        c["fa"], c["fb"], ep, torch.cuda.current_stream().cuda_stream, tg.make_options(**c["opts"]))
    assert st == tg.TG_OK, (c, tg.STATUS_NAMES.get(st, st))
    assert tg.device_error() == tg.TG_OK, c
    host = dbuf.float().cpu().numpy()
    want = ofp8.gemm_fp8_f64(A.numpy(), Bt.numpy(), c["fa"], c["fb"])
    if c["out"] == "bf16":
        want = torch.from_numpy(want).to(torch.bfloat16).double().numpy()
    mask = np.zeros(host.shape, dtype=bool)
    for b in range(batch):
        for i_ in range(M):
            lo = b * sD + i_ * ldd
            mask[lo: lo + N] = True
            assert np.array_equal(host[lo: lo + N].astype(np.float64), want[b, i_]), (c, b, i_)
    assert np.all(np.isnan(host[~mask])), ("write outside D", c)


def _case_mx(i):
    r = random.Random(7000 + i)
    M, N = r.randint(1, 600), r.randint(1, 800)
    K = 16 * r.randint(1, 70)
    batch = r.choice([1, 1, 2])
    opts = {}
    bn = r.choice([0, 128, 192, 224])
    if bn:
        opts["block_n"] = bn
    if r.random() < 0.25 and K >= 256:
        opts["split_k"] = 2
    elif r.random() < 0.2:
        opts["stream_k"] = 2
    if r.random() < 0.3:
        opts["stages"] = 2
    runs = -(-K // 32)
    return dict(M=M, N=N, K=K, batch=batch, opts=opts, fa=r.choice([0, 1]), fb=r.choice([0, 1]),
                ld_sfa=runs + r.choice([0, 0, 5]), ld_sfb=runs + r.choice([0, 3]),
                shared_sfb=batch > 1 and r.random() < 0.3, ldd_pad=r.choice([0, 3, 8]),
                seed=r.randint(0, 10 ** 6))


@pytest.mark.parametrize("i", range(24))
def test_random_mx_cases(i):
    """Block-scaled 8-bit operands: random extents (K not a multiple of 32
    included), scale pitches, shared scales, tile widths, rings and K
    splits; exact against the oracle (integer elements, scales 2^-1..2^1),
    and nothing written outside D."""
    from oracle import mx as omx

    c = _case_mx(i)
    M, N, K, batch = c["M"], c["N"], c["K"], c["batch"]
    runs = -(-K // 32)
    A = synth.make_fp8_codes((batch, M, K), c["fa"], seed=c["seed"])
    Bt = synth.make_fp8_codes((batch, N, K), c["fb"], seed=c["seed"] + 1)
    sfa = synth.make_e8m0_codes((batch, M, runs), seed=c["seed"] + 2, lo=126, hi=128)
    nb_sf = 1 if c["shared_sfb"] else batch
    sfb = synth.make_e8m0_codes((nb_sf, N, runs), seed=c["seed"] + 3, lo=126, hi=128)
    # scales in buffers with their own pitches
    fa_buf = torch.full((batch, M, c["ld_sfa"]), 255, dtype=torch.uint8)
    fa_buf[:, :, :runs] = sfa
    fb_buf = torch.full((nb_sf, N, c["ld_sfb"]), 255, dtype=torch.uint8)
    fb_buf[:, :, :runs] = sfb
    ad, bd = A.contiguous().to(dev()), Bt.contiguous().to(dev())
    fad, fbd = fa_buf.to(dev()), fb_buf.to(dev())
    ldd = N + c["ldd_pad"]
    sD = M * ldd + 8
    dbuf = torch.full(((batch - 1) * sD + M * ldd + 8,), float("nan"), dtype=torch.float32, device=dev())
    st = tg.tg_gemm_mxfp8(ad.data_ptr(), bd.data_ptr(), dbuf.data_ptr(), M, N, K, K, K, ldd, batch,
                          M * K if batch > 1 else 0, N * K if batch > 1 else 0, sD if batch > 1 else 0,
                          c["fa"], c["fb"], fad.data_ptr(), c["ld_sfa"], M * c["ld_sfa"] if batch > 1 else 0,
                          fbd.data_ptr(), c["ld_sfb"], N * c["ld_sfb"] if nb_sf > 1 else 0, None,
                          torch.cuda.current_stream().cuda_stream, tg.make_options(**c["opts"]))
    assert st == tg.TG_OK, (c, tg.STATUS_NAMES.get(st, st))
    assert tg.device_error() == tg.TG_OK, c
    host = dbuf.cpu().numpy()
    sfb_full = sfb.expand(batch, N, runs) if nb_sf == 1 else sfb
    want = omx.gemm_mx_f64(A.numpy(), Bt.numpy(), c["fa"], c["fb"], sfa.numpy(), sfb_full.numpy())
    mask = np.zeros(host.shape, dtype=bool)
    for b in range(batch):
        for i_ in range(M):
            lo = b * sD + i_ * ldd
            mask[lo: lo + N] = True
            assert np.array_equal(host[lo: lo + N].astype(np.float64), want[b, i_]), (c, b, i_)
    assert np.all(np.isnan(host[~mask])), ("write outside D", c)


def _case_mx4(i):
    r = random.Random(9000 + i)
    M, N = r.randint(1, 600), r.randint(1, 800)
    K = 32 * r.randint(1, 40)                 # whole 16-byte rows of packed elements
    k_used = K - 2 * r.randint(0, 7) if r.random() < 0.4 else K  # even K, the rest row padding
    batch = r.choice([1, 1, 2])
    opts = {}
    bn = r.choice([0, 128, 192, 224])
    if bn:
        opts["block_n"] = bn
    if r.random() < 0.25 and k_used >= 512:
        opts["split_k"] = 2
    elif r.random() < 0.2:
        opts["stream_k"] = 2
    if r.random() < 0.3 or bn == 224:
        opts["stages"] = 2
    runs = -(-k_used // 32)
    return dict(M=M, N=N, K=k_used, pitch=K, batch=batch, opts=opts, ld_sfa=runs + r.choice([0, 0, 5]),
                ld_sfb=runs + r.choice([0, 3]), shared_sfb=batch > 1 and r.random() < 0.3,
                ldd_pad=r.choice([0, 3, 8]), seed=r.randint(0, 10 ** 6))


@pytest.mark.parametrize("i", range(24))
def test_random_mxfp4_cases(i):
    """Block-scaled packed 4-bit operands: random extents (K not a multiple of
    32, rows padded past K), scale pitches, shared scales, tile widths,
    rings and K splits; exact against the oracle (all E2M1 codes, scales
    2^-1..2^1), and nothing written outside D."""
    from oracle import mx as omx

    c = _case_mx4(i)
    M, N, K, P, batch = c["M"], c["N"], c["K"], c["pitch"], c["batch"]
    runs = -(-K // 32)
    Ac = synth.make_fp4_codes((batch, M, K), seed=c["seed"])
    Bc = synth.make_fp4_codes((batch, N, K), seed=c["seed"] + 1)
    # packed rows of P elements; the padding past K holds the code of 6.0
    pad = lambda t: torch.cat([t, torch.full(t.shape[:-1] + (P - K,), 7, dtype=torch.uint8)], dim=-1)
    ad = synth.pack_fp4_codes(pad(Ac)).to(dev())
    bd = synth.pack_fp4_codes(pad(Bc)).to(dev())
    sfa = synth.make_e8m0_codes((batch, M, runs), seed=c["seed"] + 2, lo=126, hi=128)
    nb_sf = 1 if c["shared_sfb"] else batch
    sfb = synth.make_e8m0_codes((nb_sf, N, runs), seed=c["seed"] + 3, lo=126, hi=128)
    fa_buf = torch.full((batch, M, c["ld_sfa"]), 255, dtype=torch.uint8)
    fa_buf[:, :, :runs] = sfa
    fb_buf = torch.full((nb_sf, N, c["ld_sfb"]), 255, dtype=torch.uint8)
    fb_buf[:, :, :runs] = sfb
    fad, fbd = fa_buf.to(dev()), fb_buf.to(dev())
    ldd = N + c["ldd_pad"]
    sD = M * ldd + 8
    dbuf = torch.full(((batch - 1) * sD + M * ldd + 8,), float("nan"), dtype=torch.float32, device=dev())
    st = tg.tg_gemm_mxfp4(ad.data_ptr(), bd.data_ptr(), dbuf.data_ptr(), M, N, K, P, P, ldd, batch,
                          M * P if batch > 1 else 0, N * P if batch > 1 else 0, sD if batch > 1 else 0,
                          fad.data_ptr(), c["ld_sfa"], M * c["ld_sfa"] if batch > 1 else 0,
                          fbd.data_ptr(), c["ld_sfb"], N * c["ld_sfb"] if nb_sf > 1 else 0, None,
                          torch.cuda.current_stream().cuda_stream, tg.make_options(**c["opts"]))
    assert st == tg.TG_OK, (c, tg.STATUS_NAMES.get(st, st))
    assert tg.device_error() == tg.TG_OK, c
    host = dbuf.cpu().numpy()
    sfb_full = sfb.expand(batch, N, runs) if nb_sf == 1 else sfb
    want = omx.gemm_mxfp4_f64(omx.pack_fp4(Ac.numpy()), omx.pack_fp4(Bc.numpy()), K, sfa.numpy(),
                              sfb_full.numpy())
    mask = np.zeros(host.shape, dtype=bool)
    for b in range(batch):
        for i_ in range(M):
            lo = b * sD + i_ * ldd
            mask[lo: lo + N] = True
            assert np.array_equal(host[lo: lo + N].astype(np.float64), want[b, i_]), (c, b, i_)
    assert np.all(np.isnan(host[~mask])), ("write outside D", c)
