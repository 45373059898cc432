"""GPU parity of the CUDA path against the oracle, through the C ABI.

Exact-arithmetic cases use small-integer bf16 inputs (every partial sum is
an exact fp32 integer), so the GPU must equal the fp64 oracle bit for bit
whatever the tiling, ring depth, split or store path.  Random-float cases use
the contract's tolerance (relative Frobenius <= 1e-5, per element
<= 1e-5 sqrt(K) max|C|).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tiled_gemm_codegen_gb300 as tg
from gpu_helpers import assert_close, dev, oracle_dense, run

pytestmark = pytest.mark.gpu

WIDTHS = [64, 128, 192, 256]
# (tile width, cta_pair): one CTA per tile for every width, two-SM tiles
# (cluster of two CTAs, tcgen05 cta_group::2) for widths 128 and 256
CONFIGS = [(64, 1), (128, 1), (192, 1), (256, 1), (128, 2), (256, 2)]
EDGE_SHAPES = [
    (1, 1, 1), (7, 5, 3), (16, 16, 16), (17, 63, 65), (64, 64, 64), (127, 129, 128),
    (128, 128, 128), (129, 255, 257), (255, 257, 129), (200, 300, 40), (65, 513, 191),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tg.load()
    yield


def _seed(*xs):
    s = 17
    for x in xs:
        s = (s * 1000003 + int(x)) % (2 ** 31)
    return s


def _cfg_id(c):
    return f"bn{c[0]}{'-pair' if c[1] == 2 else ''}"


@pytest.mark.parametrize("cfg", CONFIGS, ids=_cfg_id)
@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_exact_integer_edge_shapes(cfg, shape):
    bn, pair = cfg
    M, N, K = shape
    A, B = synth.make_int_inputs(1, M, N, K, seed=_seed(M, N, K, bn))
    got = run(A, B, options=tg.make_options(block_n=bn, cta_pair=pair))
    assert np.array_equal(got, oracle_dense(A, B))


@pytest.mark.parametrize("cfg", CONFIGS, ids=_cfg_id)
def test_exact_integer_batched(cfg):
    bn, pair = cfg
    batch, M, N, K = 3, 131, 197, 333
    A, B = synth.make_int_inputs(batch, M, N, K, seed=_seed(batch, bn))
    got = run(A, B, options=tg.make_options(block_n=bn, cta_pair=pair))
    assert np.array_equal(got, oracle_dense(A, B))


@pytest.mark.parametrize("shape", [(197, 131, 77), (300, 200, 500), (129, 513, 1000),
                                   (1000, 64, 2048), (64, 1024, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_float_parity_default_plan(shape, dist):
    M, N, K = shape
    A, B = synth.make_inputs(1, M, N, K, dist, seed=_seed(M, N, K))
    assert_close(run(A, B), oracle_dense(A, B), K, f"{shape} {dist}")


@pytest.mark.parametrize("cfg", CONFIGS, ids=_cfg_id)
def test_float_parity_each_width(cfg):
    bn, pair = cfg
    M, N, K = 257, 389, 700
    A, B = synth.make_inputs(2, M, N, K, "normal", seed=_seed(bn, 5))
    assert_close(run(A, B, options=tg.make_options(block_n=bn, cta_pair=pair)), oracle_dense(A, B),
                 K, f"bn={bn} pair={pair}")


@pytest.mark.parametrize("bn,pair,depths", [(64, 1, [2, 4, 6, 8]), (128, 1, [2, 3, 4, 6]),
                                            (192, 1, [2, 3, 4]), (256, 1, [2, 3, 4]),
                                            (128, 2, [2, 4, 8]), (256, 2, [2, 4, 6])])
def test_ring_depth_bitwise_invariance(bn, pair, depths):
    """OCANNL pipeline_depth: the pipelined rendering reads the same values in
    the same order, so the output is bitwise independent of the depth."""
    M, N, K = 300, 520, 1100
    A, B = synth.make_inputs(1, M, N, K, "uniform", seed=_seed(bn, 7))
    outs = [run(A, B, options=tg.make_options(block_n=bn, stages=s, cta_pair=pair)) for s in depths]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    assert_close(outs[0], oracle_dense(A, B), K)


@pytest.mark.parametrize("pair", [1, 2])
def test_persistent_grid_bitwise_invariance(pair):
    """A CTA (or CTA pair) that walks many tiles (accumulator double buffer,
    ring phases wrapping) gives the same bits as one tile per worker."""
    M, N, K = 640, 768, 512
    A, B = synth.make_inputs(1, M, N, K, "normal", seed=3)
    base = run(A, B, options=tg.make_options(block_n=128, cta_pair=pair))
    for ctas in (2, 6, 14):
        got = run(A, B, options=tg.make_options(block_n=128, max_ctas=ctas, cta_pair=pair))
        assert np.array_equal(got, base), ctas


def test_pair_tiles_equal_single_tiles_exactly():
    """Two-SM tiles and one-CTA tiles compute the same exact sums."""
    M, N, K = 513, 600, 700
    A, B = synth.make_int_inputs(1, M, N, K, seed=77)
    one = run(A, B, options=tg.make_options(block_n=256, cta_pair=1))
    two = run(A, B, options=tg.make_options(block_n=256, cta_pair=2))
    assert np.array_equal(one, two)
    assert np.array_equal(two, oracle_dense(A, B))


@pytest.mark.parametrize("bn,pair", [(192, 1), (256, 2)])
def test_epilogue_paths_bitwise_equal(bn, pair):
    M, N, K = 333, 444, 555
    A, B = synth.make_inputs(1, M, N, K, "uniform", seed=4)
    t = run(A, B, options=tg.make_options(block_n=bn, epilogue=1, cta_pair=pair))
    d = run(A, B, options=tg.make_options(block_n=bn, epilogue=2, cta_pair=pair))
    assert np.array_equal(t, d)
    assert_close(t, oracle_dense(A, B), K)


def test_pack_path_bitwise_equal():
    M, N, K = 190, 250, 310
    A, B = synth.make_inputs(1, M, N, K, "normal", seed=5)
    plain = run(A, B, options=tg.make_options(block_n=128))
    packed = run(A, B, options=tg.make_options(block_n=128, force_pack=1))
    assert np.array_equal(plain, packed)


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("splits", [2, 3, 4, 7])
def test_split_k_exact_integer(splits, pair):
    """Split reduction: the combined partials equal the full sum exactly
    with integer inputs."""
    M, N, K = 150, 300, 2048
    A, B = synth.make_int_inputs(1, M, N, K, seed=splits)
    got = run(A, B, options=tg.make_options(block_n=128, split_k=splits, cta_pair=pair))
    assert np.array_equal(got, oracle_dense(A, B))


def test_split_k_deterministic_and_close():
    """Deterministic per plan (bitwise run to run), within tolerance of the
    oracle and of other split factors (OCANNL two-pass split reduction)."""
    M, N, K = 64, 2048, 8192
    A, B = synth.make_inputs(1, M, N, K, "normal002", seed=9)
    ref = oracle_dense(A, B)
    outs = {}
    for s in (1, 2, 4, 8):
        o1 = run(A, B, options=tg.make_options(block_n=256, split_k=s))
        o2 = run(A, B, options=tg.make_options(block_n=256, split_k=s))
        assert np.array_equal(o1, o2), s
        assert_close(o1, ref, K, f"split {s}")
        outs[s] = o1


def test_split_k_batched_ragged():
    batch, M, N, K = 3, 100, 300, 1000
    A, B = synth.make_int_inputs(batch, M, N, K, seed=12)
    got = run(A, B, options=tg.make_options(block_n=64, split_k=5, max_ctas=4))
    assert np.array_equal(got, oracle_dense(A, B))


def _guarded_c(M, N, ldc, rows_pad=3, lead=0):
    """A NaN-filled device buffer and a view C[M, N] with row stride ldc
    starting `lead` elements in."""
    total = lead + (M + rows_pad) * ldc
    buf = torch.full((total,), float("nan"), dtype=torch.float32, device=dev())
    view = buf[lead: lead + M * ldc].view(M, ldc)[:, :N]
    return buf, view


@pytest.mark.parametrize("ldc_pad,lead", [(0, 0), (24, 0), (3, 0), (8, 1), (5, 3)])
def test_guard_bands(ldc_pad, lead):
    """Elements of C outside the M x N block (row padding, trailing rows,
    leading elements) are never written; covers both store paths."""
    M, N, K = 150, 200, 96
    ldc = N + ldc_pad
    A, B = synth.make_int_inputs(1, M, N, K, seed=ldc_pad)
    buf, C = _guarded_c(M, N, ldc, lead=lead)
    tg.gemm(A.to(dev()), B.to(dev()), C)
    assert tg.device_error() == tg.TG_OK
    host = buf.cpu().numpy()
    mask = np.zeros(host.shape, dtype=bool)
    for i in range(M):
        mask[lead + i * ldc: lead + i * ldc + N] = True
    assert np.all(np.isnan(host[~mask])), "write outside the M x N block"
    got = np.stack([host[lead + i * ldc: lead + i * ldc + N] for i in range(M)]).astype(np.float64)
    assert np.array_equal(got, oracle_dense(A, B))


@pytest.mark.parametrize("a_off,b_off,lda_pad,ldb_pad", [(1, 0, 0, 0), (0, 3, 0, 0), (0, 0, 1, 0),
                                                          (0, 0, 0, 5), (2, 1, 3, 7)])
def test_misaligned_operands_use_pack(a_off, b_off, lda_pad, ldb_pad):
    M, N, K = 97, 211, 150
    lda, ldb = K + lda_pad, N + ldb_pad
    Ai, Bi = synth.make_int_inputs(1, M, N, K, seed=a_off * 10 + b_off)
    abuf = torch.zeros(a_off + M * lda, dtype=torch.bfloat16)
    bbuf = torch.zeros(b_off + K * ldb, dtype=torch.bfloat16)
    abuf[a_off:].view(M, lda)[:, :K] = Ai
    bbuf[b_off:].view(K, ldb)[:, :N] = Bi
    ad = abuf.to(dev())
    bd = bbuf.to(dev())
    A = ad[a_off:].view(M, lda)[:, :K]
    B = bd[b_off:].view(K, ldb)[:, :N]
    C = torch.empty(M, N, dtype=torch.float32, device=dev())
    # the persistent kernel (the planner would take the direct-load kernel
    # for a problem this small)
    opts = tg.make_options(direct=1)
    info = tg.plan(M, N, K, lda=lda, ldb=ldb, A=A.data_ptr(), B=B.data_ptr(), C=C.data_ptr(), options=opts)
    assert info["pack_a"] == int(a_off % 8 != 0 or lda % 8 != 0)
    assert info["pack_b"] == int(b_off % 8 != 0 or ldb % 8 != 0)
    tg.gemm(A, B, C, options=opts)
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(Ai, Bi))


@pytest.mark.parametrize("direct", [1, 2], ids=["persistent", "direct"])
@pytest.mark.parametrize("a_off,b_off,lda_pad,ldb_pad,M,N,K", [
    (1, 7, 0, 0, 131, 257, 300),     # every row start misaligned, odd ld
    (0, 0, 0, 1, 64, 95, 4100),      # A rows alternate 8- and 16-byte alignment
    (3, 5, 2, 3, 5, 9, 7),           # rows shorter than one 16-byte chunk
    (0, 2, 0, 1, 33, 1031, 1031),    # a ragged last chunk in every row
])
def test_pack_reads_nothing_outside_rows(a_off, b_off, lda_pad, ldb_pad, M, N, K, direct):
    """Every element around and between the operands' rows is NaN: the
    realigning pack reads whole aligned 16-byte blocks, so a stray byte
    shifted into a packed row, or a tail not masked, would turn outputs
    into NaN; the direct-load kernel reads the rows in place, element by
    element.  Integer inputs make the product exact."""
    lda, ldb = K + lda_pad, N + ldb_pad
    Ai, Bi = synth.make_int_inputs(1, M, N, K, seed=M + N)
    nan = float("nan")
    abuf = torch.full((a_off + M * lda + 16,), nan, dtype=torch.bfloat16)
    bbuf = torch.full((b_off + K * ldb + 16,), nan, dtype=torch.bfloat16)
    abuf[a_off:a_off + M * lda].view(M, lda)[:, :K] = Ai
    bbuf[b_off:b_off + K * ldb].view(K, ldb)[:, :N] = Bi
    ad, bd = abuf.to(dev()), bbuf.to(dev())
    A = ad[a_off:a_off + M * lda].view(M, lda)[:, :K]
    B = bd[b_off:b_off + K * ldb].view(K, ldb)[:, :N]
    C = torch.empty(M, N, dtype=torch.float32, device=dev())
    tg.gemm(A, B, C, options=tg.make_options(direct=direct))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(C.cpu().double().numpy(), oracle_dense(Ai, Bi))


def test_strided_batches_with_gaps():
    batch, M, N, K = 4, 70, 90, 110
    Ai, Bi = synth.make_int_inputs(batch, M, N, K, seed=21)
    sA, sB = M * K + 64, K * N + 40
    abuf = torch.zeros(batch * sA, dtype=torch.bfloat16)
    bbuf = torch.zeros(batch * sB, dtype=torch.bfloat16)
    for b in range(batch):
        abuf[b * sA: b * sA + M * K] = Ai[b].reshape(-1)
        bbuf[b * sB: b * sB + K * N] = Bi[b].reshape(-1)
    ad, bd = abuf.to(dev()), bbuf.to(dev())
    A = torch.as_strided(ad, (batch, M, K), (sA, K, 1))
    B = torch.as_strided(bd, (batch, K, N), (sB, N, 1))
    got = tg.gemm(A, B)
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(got.cpu().double().numpy(), oracle_dense(Ai, Bi))


def test_broadcast_operand():
    """Batch stride 0: the same B for every problem."""
    batch, M, N, K = 5, 130, 140, 150
    Ai, _ = synth.make_int_inputs(batch, M, N, K, seed=31)
    _, Bi = synth.make_int_inputs(1, M, N, K, seed=32)
    got = tg.gemm(Ai.to(dev()), Bi.to(dev()))
    assert tg.device_error() == tg.TG_OK
    ref = oracle_dense(Ai, Bi.unsqueeze(0).expand(batch, K, N).contiguous())
    assert np.array_equal(got.cpu().double().numpy(), ref)


def test_broadcast_a_and_many_tiny_problems():
    """A shared across the batch (stride 0); and 3000 tiny problems (one
    tile each, far more units than workers: the persistent schedule's
    strided walk over problems), both exact, under each tile form."""
    batch, M, N, K = 4, 150, 260, 300
    _, Bi = synth.make_int_inputs(batch, M, N, K, seed=33)
    Ai, _ = synth.make_int_inputs(1, M, N, K, seed=34)
    got = tg.gemm(Ai.to(dev()), Bi.to(dev()))
    assert tg.device_error() == tg.TG_OK
    ref = oracle_dense(Ai.unsqueeze(0).expand(batch, M, K).contiguous(), Bi)
    assert np.array_equal(got.cpu().double().numpy(), ref)
    batch, M, N, K = 3000, 9, 17, 40
    Ai, Bi = synth.make_int_inputs(batch, M, N, K, seed=35)
    ref = oracle_dense(Ai, Bi)
    Ad, Bd = Ai.to(dev()), Bi.to(dev())
    for opts in ({}, {"block_n": 64}, {"block_n": 256, "cta_pair": 2}, {"split_k": 1, "max_ctas": 7}):
        got = tg.gemm(Ad, Bd, options=tg.make_options(**opts))
        assert tg.device_error() == tg.TG_OK
        assert np.array_equal(got.cpu().double().numpy(), ref), opts


def test_k_zero_and_empty():
    C = torch.full((5, 6), 7.0, device=dev())
    A = torch.empty(5, 0, dtype=torch.bfloat16, device=dev())
    B = torch.empty(0, 6, dtype=torch.bfloat16, device=dev())
    tg.gemm(A, B, C)
    assert tg.device_error() == tg.TG_OK
    assert torch.all(C.cpu() == 0)
    # M == 0: nothing enqueued, status OK
    A0 = torch.empty(0, 4, dtype=torch.bfloat16, device=dev())
    B0 = torch.ones(4, 3, dtype=torch.bfloat16, device=dev())
    C0 = tg.gemm(A0, B0)
    assert C0.shape == (0, 3)


def test_host_entry_point_matches_device():
    M, N, K = 210, 170, 390
    A, B = synth.make_inputs(1, M, N, K, "uniform", seed=41)
    ch = tg.gemm_host(A.pin_memory(), B.pin_memory())
    cd = run(A, B)
    assert np.array_equal(ch.double().numpy(), cd)
    # gaps between rows of a host C are preserved
    ldc = N + 6
    Cbuf = torch.full((M, ldc), -3.0)
    tg.gemm_host(A, B, Cbuf[:, :N])
    assert torch.all(Cbuf[:, N:] == -3.0)
    assert np.array_equal(Cbuf[:, :N].double().numpy(), cd)


def test_watchdog_reports_timeout_and_recovers():
    """A wait on a barrier nothing completes: the kernel gives up after the
    limit, records the error and exits; the host reads TG_ERR_TIMEOUT, the
    word is cleared, and the next call is exact again."""
    M, N, K = 300, 300, 256
    A, B = synth.make_int_inputs(1, M, N, K, seed=51)
    ad, bd = A.to(dev()), B.to(dev())
    # one tile per CTA, one CTA walking all tiles, and the same for CTA pairs
    for ctas, pair in ((0, 1), (1, 1), (0, 2), (2, 2)):
        opts = tg.make_options(debug_stall=1, timeout_ns=20_000_000, block_n=128, max_ctas=ctas,
                               cta_pair=pair)
        tg.gemm(ad, bd, options=opts)
        assert tg.device_error() == tg.TG_ERR_TIMEOUT
        assert tg.device_error() == tg.TG_OK
    got = tg.gemm(ad, bd)
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(got.cpu().double().numpy(), oracle_dense(A, B))


def test_split_k_counters_reset_after_timeout():
    """An aborted split-K launch leaves the counters part-way; reading the
    error resets them, so the next split-K call is exact."""
    M, N, K = 128, 256, 1024
    A, B = synth.make_int_inputs(1, M, N, K, seed=61)
    ad, bd = A.to(dev()), B.to(dev())
    tg.gemm(ad, bd, options=tg.make_options(debug_stall=1, timeout_ns=20_000_000, split_k=4))
    assert tg.device_error() == tg.TG_ERR_TIMEOUT
    got = tg.gemm(ad, bd, options=tg.make_options(split_k=4))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(got.cpu().double().numpy(), oracle_dense(A, B))


def test_invalid_arguments_on_device():
    A = torch.zeros(4, 4, dtype=torch.bfloat16, device=dev())
    B = torch.zeros(4, 4, dtype=torch.bfloat16, device=dev())
    C = torch.zeros(4, 4, dtype=torch.float32, device=dev())
    # C overlapping A
    st = tg.tg_gemm(A.data_ptr(), B.data_ptr(), A.data_ptr(), 4, 4, 4, 4, 4, 4, 1, 16, 16, 16)
    assert st == tg.TG_ERR_INVALID_ARG
    # bad override
    st = tg.tg_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), 4, 4, 4, 4, 4, 4, 1, 16, 16, 16,
                       None, tg.make_options(block_n=96))
    assert st == tg.TG_ERR_INVALID_ARG
    st = tg.tg_gemm_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), 4, 4, 4, 4, 4, 4, 1, 16, 16, 16,
                       None, tg.make_options(stages=5, block_n=256))
    assert st == tg.TG_ERR_INVALID_ARG


def test_plan_queries_device():
    info = tg.plan(4096, 4096, 4096)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 1 <= info["grid"] <= sms


@pytest.mark.parametrize("bn,pair,ctas,shape", [
    (128, 1, 7, (1000, 1000, 2048)),   # 64 tiles on 7 CTAs: 1 tile split 7 ways
    (64, 1, 5, (300, 700, 1000)),      # ragged tiles and k-blocks
    (256, 2, 6, (1000, 900, 1500)),    # two-SM tiles on 3 pairs
    (128, 2, 10, (777, 1300, 640)),
    (128, 1, 7, (1000, 1000, 64)),     # one k-block: most ranges empty
])
def test_stream_k_exact_integer(bn, pair, ctas, shape):
    """Stream-K: whole-tile waves, then shared k-block ranges combined in k
    order; exact with integer inputs, and bitwise run to run."""
    M, N, K = shape
    A, B = synth.make_int_inputs(2 if bn == 64 else 1, M, N, K, seed=_seed(M, N, K, ctas))
    opts = tg.make_options(block_n=bn, cta_pair=pair, max_ctas=ctas, stream_k=2)
    info = tg.plan(M, N, K, 2 if bn == 64 else 1, sm_count=152, options=opts)
    assert info["stream_k"] == 2 and info["sk_tiles"] > 0
    got = run(A, B, options=opts)
    assert np.array_equal(got, oracle_dense(A, B))
    assert np.array_equal(run(A, B, options=opts), got)


def test_stream_k_float_deterministic_and_close():
    M, N, K = 1100, 1500, 3000
    A, B = synth.make_inputs(1, M, N, K, "normal", seed=91)
    opts = tg.make_options(block_n=256, cta_pair=2, max_ctas=10, stream_k=2)
    o1 = run(A, B, options=opts)
    o2 = run(A, B, options=opts)
    assert np.array_equal(o1, o2)
    ref = oracle_dense(A, B)
    assert_close(o1, ref, K, "stream-K")
    off = run(A, B, options=tg.make_options(block_n=256, cta_pair=2, max_ctas=10, stream_k=1))
    assert_close(off, ref, K, "stream-K off")


def test_stream_k_watchdog():
    M, N, K = 1000, 1000, 2048
    A, B = synth.make_int_inputs(1, M, N, K, seed=93)
    ad, bd = A.to(dev()), B.to(dev())
    tg.gemm(ad, bd, options=tg.make_options(debug_stall=1, timeout_ns=20_000_000, block_n=128,
                                            max_ctas=7, stream_k=2))
    assert tg.device_error() == tg.TG_ERR_TIMEOUT
    got = tg.gemm(ad, bd, options=tg.make_options(block_n=128, max_ctas=7, stream_k=2))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(got.cpu().double().numpy(), oracle_dense(A, B))


def _stored(t_logical, col_major, pad=0, offset=0):
    """Device copy of a logical [batch?, rows, cols] bf16 matrix in row- or
    column-major storage with `pad` extra elements per stored row and an
    element offset from an allocation start.  Returns (view, ld)."""
    t = t_logical if t_logical.dim() == 3 else t_logical.unsqueeze(0)
    batch, rows, cols = t.shape
    srows, scols = (cols, rows) if col_major else (rows, cols)
    ld = scols + pad
    per = srows * ld
    buf = torch.zeros(offset + batch * per, dtype=torch.bfloat16)
    for b in range(batch):
        block = buf[offset + b * per: offset + (b + 1) * per].view(srows, ld)
        block[:, :scols] = t[b].t() if col_major else t[b]
    d = buf.to(dev())
    if col_major:
        v = torch.as_strided(d, (batch, rows, cols), (per, 1, ld), offset)
    else:
        v = torch.as_strided(d, (batch, rows, cols), (per, ld, 1), offset)
    return (v if t_logical.dim() == 3 else v[0]), ld


@pytest.mark.parametrize("a_cm,b_cm", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("cfg", [(128, 1), (256, 1), (256, 2), (128, 2), (64, 1), (192, 1)], ids=_cfg_id)
def test_transposed_layouts_exact(a_cm, b_cm, cfg):
    """Column-major A (stored K x M) and/or B (stored N x K): K-major and
    MN-major shared-memory atoms swap roles; exact with integer inputs."""
    bn, pair = cfg
    M, N, K = 277, 389, 333
    A, B = synth.make_int_inputs(1, M, N, K, seed=_seed(a_cm, b_cm, bn, pair))
    Ad, lda = _stored(A, a_cm)
    Bd, ldb = _stored(B, b_cm)
    got = tg.gemm(Ad, Bd, options=tg.make_options(block_n=bn, cta_pair=pair))
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(got.cpu().double().numpy(), oracle_dense(A, B))


@pytest.mark.parametrize("a_cm,b_cm", [(1, 0), (0, 1), (1, 1)])
def test_transposed_batched_split_stream_and_pack(a_cm, b_cm):
    batch, M, N, K = 3, 190, 300, 1000
    A, B = synth.make_int_inputs(batch, M, N, K, seed=a_cm * 2 + b_cm)
    ref = oracle_dense(A, B)
    for pad, off, extra in [(0, 0, dict(split_k=3)), (8, 0, dict(stream_k=2, max_ctas=7)),
                            (3, 1, dict()), (0, 0, dict(cta_pair=2, block_n=256, stream_k=2, max_ctas=10))]:
        Ad, _ = _stored(A, a_cm, pad=pad, offset=off)
        Bd, _ = _stored(B, b_cm, pad=pad, offset=off)
        got = tg.gemm(Ad, Bd, options=tg.make_options(**extra))
        assert tg.device_error() == tg.TG_OK
        assert np.array_equal(got.cpu().double().numpy(), ref), (pad, off, extra)


def test_transposed_float_and_fused():
    M, N, K = 300, 260, 777
    A, B = synth.make_inputs(1, M, N, K, "normal", seed=17)
    At = A.t().contiguous().to(dev()).t()   # column-major view
    Bt = B.t().contiguous().to(dev()).t()
    got = tg.gemm(At, Bt)
    assert tg.device_error() == tg.TG_OK
    assert_close(got.cpu().double().numpy(), oracle_dense(A, B), K)
    plain = tg.gemm(A.to(dev()), B.to(dev()))
    fused = tg.gemm_fused(At, Bt, activation="relu")
    assert tg.device_error() == tg.TG_OK
    assert np.array_equal(fused.cpu().numpy(), np.maximum(plain.cpu().numpy(), 0))


def test_transposed_host_entry():
    M, N, K = 150, 170, 190
    A, B = synth.make_int_inputs(1, M, N, K, seed=23)
    At = A.t().contiguous()
    Bt = B.t().contiguous()
    C = torch.zeros(M, N)
    st = tg.tg_gemm_host(At.data_ptr(), Bt.data_ptr(), C.data_ptr(), M, N, K, M, K, N, 1, 0, 0, 0,
                         torch.cuda.current_stream().cuda_stream,
                         tg.make_options(a_col_major=1, b_col_major=1))
    assert st == tg.TG_OK
    assert np.array_equal(C.double().numpy(), oracle_dense(A, B))


def _host_strided(rows, cols, ld, fill=float("nan")):
    """A host bf16 buffer of `rows` rows of pitch `ld` and a view of its
    rows x cols block."""
    buf = torch.full((rows * ld,), fill, dtype=torch.bfloat16)
    return buf, buf.view(rows, ld)[:, :cols]


@pytest.mark.parametrize("M,N,K,lda_pad,ldb_pad,ldc_pad", [
    (2048, 256, 300, 0, 0, 0),     # A the larger operand: streamed in pieces of rows
    (1031, 300, 200, 3, 5, 7),     # row pieces, host rows not 16-byte aligned, C row gaps
    (100, 3000, 200, 1, 0, 2),     # B the larger operand: streamed in pieces of columns
    (64, 1300, 520, 0, 3, 1),      # column pieces with a ragged last piece
])
def test_host_entry_pipelined_pieces(M, N, K, lda_pad, ldb_pad, ldc_pad):
    """tg_gemm_host stages the operands with 16-byte row pitches and
    multiplies piece by piece while copies overlap: exact integer products,
    and the host C keeps every element outside the M x N block."""
    Ai, Bi = synth.make_int_inputs(1, M, N, K, seed=M + 7 * N)
    lda, ldb, ldc = K + lda_pad, N + ldb_pad, N + ldc_pad
    _, A = _host_strided(M, K, lda)
    _, B = _host_strided(K, N, ldb)
    A.copy_(Ai)
    B.copy_(Bi)
    cbuf = torch.full((M * ldc,), float("nan"), dtype=torch.float32)
    C = cbuf.view(M, ldc)[:, :N]
    tg.gemm_host(A, B, C)
    assert np.array_equal(C.double().numpy(), oracle_dense(Ai, Bi))
    if ldc_pad:
        assert torch.all(torch.isnan(cbuf.view(M, ldc)[:, N:]))


def test_host_entry_pipelined_batches():
    """Batched host operands with gaps between problems: pieces of problems."""
    batch, M, N, K = 11, 70, 90, 110
    Ai, Bi = synth.make_int_inputs(batch, M, N, K, seed=99)
    sA, sB, sC = M * K + 24, K * N + 8, M * N + 40
    abuf = torch.full((batch * sA,), float("nan"), dtype=torch.bfloat16)
    bbuf = torch.full((batch * sB,), float("nan"), dtype=torch.bfloat16)
    cbuf = torch.full((batch * sC,), float("nan"), dtype=torch.float32)
    for b in range(batch):
        abuf[b * sA: b * sA + M * K] = Ai[b].reshape(-1)
        bbuf[b * sB: b * sB + K * N] = Bi[b].reshape(-1)
    st = tg.tg_gemm_host(abuf.data_ptr(), bbuf.data_ptr(), cbuf.data_ptr(), M, N, K, K, N, N, batch,
                         sA, sB, sC, torch.cuda.current_stream().cuda_stream, None)
    assert st == tg.TG_OK
    want = oracle_dense(Ai, Bi)
    for b in range(batch):
        got = cbuf[b * sC: b * sC + M * N].view(M, N).double().numpy()
        assert np.array_equal(got, want[b]), b
        assert torch.all(torch.isnan(cbuf[b * sC + M * N: (b + 1) * sC]))


@pytest.mark.parametrize("M,N,K,a_cm,b_cm", [(1500, 200, 300, 1, 0), (90, 1800, 250, 0, 1),
                                             (1100, 150, 260, 1, 1)])
def test_host_entry_pipelined_transposed(M, N, K, a_cm, b_cm):
    """Column-major operands through the host entry point, with pieces of
    rows (A streamed) or columns (B streamed)."""
    Ai, Bi = synth.make_int_inputs(1, M, N, K, seed=M + N + a_cm)
    A = Ai.t().contiguous() if a_cm else Ai.contiguous()
    B = Bi.t().contiguous() if b_cm else Bi.contiguous()
    lda = M if a_cm else K
    ldb = K if b_cm else N
    C = torch.full((M, N), float("nan"))
    st = tg.tg_gemm_host(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, N, 1, 0, 0, 0,
                         torch.cuda.current_stream().cuda_stream,
                         tg.make_options(a_col_major=a_cm, b_col_major=b_cm))
    assert st == tg.TG_OK
    assert np.array_equal(C.double().numpy(), oracle_dense(Ai, Bi))


def test_host_entry_empty_sum():
    """K == 0 through the host entry point: C is all zeros."""
    M, N = 37, 45
    A = torch.empty(M, 0, dtype=torch.bfloat16)
    B = torch.empty(0, N, dtype=torch.bfloat16)
    C = torch.full((M, N), float("nan"))
    tg.gemm_host(A, B, C)
    assert torch.all(C == 0)


@pytest.mark.parametrize("direct", [1, 2], ids=["persistent", "direct"])
@pytest.mark.parametrize("N", [423, 422, 421, 420])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_store_never_writes_row_padding(N, out, direct):
    """C rows 16-byte aligned (the persistent kernel's tensor-memory-
    accelerator store path; the direct-load kernel's plain stores) but N not
    ending on a 16-byte boundary: the padding between rows stays untouched
    (a TMA store clips only at 16-byte granularity)."""
    M, K = 70, 64
    A, B = synth.make_int_inputs(1, M, N, K, seed=N)
    ldc = (N + 8) // 8 * 8 + 8
    dt = torch.float32 if out == "f32" else torch.bfloat16
    buf = torch.full((M * ldc,), float("nan"), dtype=dt, device=dev())
    D = buf.view(M, ldc)[:, :N]
    opts = tg.make_options(direct=direct)
    if out == "f32":
        tg.gemm(A.to(dev()), B.to(dev()), D, options=opts)
    else:
        tg.gemm_fused(A.to(dev()), B.to(dev()), D, options=opts)
    assert tg.device_error() == tg.TG_OK
    host = buf.view(M, ldc).float().cpu().numpy()
    assert np.all(np.isnan(host[:, N:])), "write into the row padding"
    want = oracle_dense(A, B)
    got = host[:, :N].astype(np.float64)
    if out == "f32":
        assert np.array_equal(got, want)
    else:
        assert np.array_equal(got, torch.from_numpy(want).to(torch.bfloat16).double().numpy())


# Outputs of at most 64 rows take ring slots of 64 rows of A (8 slots at
# width 128, 6 at width 192); the MMA reads the upper 64 rows from the memory
# after the slot and their accumulator rows are never stored.
HALF_A_SHAPES = [(1, 129, 64), (5, 700, 77), (33, 257, 300), (64, 1000, 1000), (64, 192, 4100)]


@pytest.mark.parametrize("bn", [128, 192])
@pytest.mark.parametrize("shape", HALF_A_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_half_height_a_exact(bn, shape):
    M, N, K = shape
    info = tg.plan(M, N, K, sm_count=152, options=tg.make_options(block_n=bn))
    assert info["block_m"] == 64 and info["stages"] == (8 if bn == 128 else 6)
    A, B = synth.make_int_inputs(1, M, N, K, seed=_seed(M, N, K, bn, 64))
    got = run(A, B, options=tg.make_options(block_n=bn))
    assert np.array_equal(got, oracle_dense(A, B))


@pytest.mark.parametrize("bn", [128, 192])
@pytest.mark.parametrize("layout", ["nn", "tn", "nt", "tt"])
def test_half_height_a_bitwise_equals_full_slots(bn, layout):
    """The same tile and k order with 64-row A slots and with 128-row ones
    (an explicit shallower ring): bitwise equal, for every operand layout,
    batched and with a K split."""
    b, M, N, K = 3, 50, 517, 1100
    gen = torch.Generator().manual_seed(_seed(b, M, N, K, bn))
    A = torch.randn(b, M, K, generator=gen).to(torch.bfloat16).to(dev())
    B = torch.randn(b, K, N, generator=gen).to(torch.bfloat16).to(dev())
    if layout[0] == "t":
        A = A.transpose(-1, -2).contiguous().transpose(-1, -2)
    if layout[1] == "t":
        B = B.transpose(-1, -2).contiguous().transpose(-1, -2)
    for split in (1, 3):
        half = tg.gemm(A, B, options=tg.make_options(block_n=bn, split_k=split))
        full = tg.gemm(A, B, options=tg.make_options(block_n=bn, split_k=split, stages=4))
        assert tg.device_error() == tg.TG_OK
        assert torch.equal(half, full)
    ref = oracle.gemm_dense_f64(A.cpu(), B.cpu())
    assert_close(half.cpu().double().numpy(), ref, K)


@pytest.mark.parametrize("bn", [128, 192])
def test_half_height_a_fp8_bitwise_equals_full_slots(bn):
    M, N, K = 64, 28672 // 8, 2048
    A = synth.make_fp8_codes((M, K), 0, seed=_seed(M, K, bn), kind="normal").to(dev()).view(torch.float8_e4m3fn)
    Bt = synth.make_fp8_codes((N, K), 0, seed=_seed(N, K, bn), kind="normal").to(dev()).view(torch.float8_e4m3fn)
    info = tg.plan(M, N, K, sm_count=152, operands="fp8", options=tg.make_options(block_n=bn))
    assert info["block_m"] == 64
    half = tg.gemm_fp8(A, Bt, options=tg.make_options(block_n=bn))
    full = tg.gemm_fp8(A, Bt, options=tg.make_options(block_n=bn, stages=4))
    assert tg.device_error() == tg.TG_OK
    assert torch.equal(half, full)
