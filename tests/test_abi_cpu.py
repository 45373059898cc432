"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point the header declares, its structs match the header's
layout, and its host logic (argument checks, planner) behaves as documented.
No call here reaches the GPU: validation and tg_plan(sm_count > 0) run
before (and without) any CUDA call."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import synth
import tiled_gemm_codegen_gb300 as tg
from tiled_gemm_codegen_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg_gemm.h")


@pytest.fixture(scope="module")
def lib():
    return _abi.load(build_if_missing=True)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) == set(_abi.SIGNATURES), names
    for name in names:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    assert {n for n in exported if not n.startswith("_")} == set(names), "unexpected exports"


def test_struct_layout_matches_header():
    src = r"""
#include <stddef.h>
#include <stdio.h>
#include "tg_gemm.h"
int main(void) {
  printf("%zu %zu %zu %zu\n", sizeof(tg_options), offsetof(tg_options, timeout_ns),
         offsetof(tg_options, debug_stall), sizeof(tg_plan_info));
  printf("%zu %zu %zu\n", offsetof(tg_plan_info, num_units), offsetof(tg_plan_info, grid),
         offsetof(tg_plan_info, workspace_bytes));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                               check=True).stdout.split()]
    O, P = _abi.tg_options, _abi.tg_plan_info
    assert vals == [ctypes.sizeof(O), O.timeout_ns.offset, O.debug_stall.offset, ctypes.sizeof(P),
                    P.num_units.offset, P.grid.offset, P.workspace_bytes.offset]


def test_status_strings(lib):
    for code in range(6):
        assert tg.tg_status_string(code)
    assert tg.tg_status_string(99) == "unknown status"


A0, B0, C0 = 0x10000, 0x20000000, 0x40000000  # placeholder addresses, never dereferenced


@pytest.mark.parametrize("args", [
    dict(M=-1), dict(N=-2), dict(K=-3), dict(batch=0), dict(lda=3), dict(ldb=4), dict(ldc=5),
    dict(M=2 ** 31), dict(A=0), dict(B=0), dict(C=0), dict(strideA=-1),
    dict(batch=2, strideC=10),                  # problems overlap in C
    dict(C=A0 + 8),                             # C overlaps A
    dict(C=B0),                                 # C overlaps B
    dict(lda=2 ** 41),
])
def test_invalid_arguments_rejected_before_any_cuda_call(lib, args):
    base = dict(A=A0, B=B0, C=C0, M=8, N=8, K=8, lda=8, ldb=8, ldc=8, batch=1,
                strideA=64, strideB=64, strideC=64)
    base.update(args)
    st = tg.tg_gemm(base["A"], base["B"], base["C"], base["M"], base["N"], base["K"], base["lda"],
                    base["ldb"], base["ldc"], base["batch"], base["strideA"], base["strideB"],
                    base["strideC"], None)
    assert st == tg.TG_ERR_INVALID_ARG


def test_column_major_leading_dimensions(lib):
    """With column-major storage the leading dimension bounds the stored
    row: lda >= M for A stored K x M, ldb >= K for B stored N x K."""
    base = [A0, B0, C0, 8, 6, 4]
    ok = tg.make_options(a_col_major=1, b_col_major=1)
    # lda = 8 >= M, ldb = 4 >= K: plan accepted (host-only planning)
    st, _ = tg.tg_plan(*base, 8, 4, 6, 1, 32, 24, 48, 152, ok)
    assert st == tg.TG_OK
    st, _ = tg.tg_plan(*base, 7, 4, 6, 1, 32, 24, 48, 152, ok)
    assert st == tg.TG_ERR_INVALID_ARG
    st, _ = tg.tg_plan(*base, 8, 3, 6, 1, 32, 24, 48, 152, ok)
    assert st == tg.TG_ERR_INVALID_ARG


def test_empty_output_is_ok_without_gpu(lib):
    assert tg.tg_gemm(0, 0, 0, 0, 5, 7, 7, 5, 5, 1, 0, 0, 0, None) == tg.TG_OK
    assert tg.tg_gemm(0, 0, 0, 5, 0, 7, 7, 0, 0, 1, 0, 0, 0, None) == tg.TG_OK


def _plan(w, **kw):
    return tg.plan(w.M, w.N, w.K, w.batch, sm_count=152, **kw)


def test_plan_of_each_workload(lib):
    for w in synth.WORKLOADS.values():
        info = _plan(w)
        if info["direct"] == 2:
            # small problem: the direct-load kernel, one CTA per 128 x 64 tile
            assert w.name == "ragged_197x131x77"
            assert (info["block_m"], info["block_n"], info["block_k"]) == (128, 64, 64)
            assert info["grid"] == info["num_units"] == w.batch * -(-w.M // 128) * -(-w.N // 64)
            assert info["stages"] == min(4, -(-w.K // 64)) and info["tmem_cols"] == 64
            assert info["pack_a"] == info["pack_b"] == 0 and info["workspace_bytes"] == 0
            assert info["epilogue"] == 2 and info["split_k"] == 1 and info["smem_bytes"] <= 232448
            continue
        assert info["direct"] == 1
        assert info["block_k"] == 64 and info["cta_pair"] in (1, 2)
        # outputs of at most 64 rows: ring slots of 64 rows of A
        assert info["block_m"] == (64 if w.M <= 64 and info["cta_pair"] == 1 else 128 * info["cta_pair"])
        assert info["tiles_m"] == -(-w.M // info["block_m"])
        if info["cta_pair"] == 2:
            assert info["block_n"] in (128, 256) and info["grid"] % 2 == 0
        assert info["tiles_n"] == -(-w.N // info["block_n"])
        assert info["k_blocks"] == -(-w.K // 64)
        assert info["num_units"] == w.batch * info["tiles_m"] * info["tiles_n"] * info["split_k"]
        assert 1 <= info["grid"] <= 152 and info["grid"] <= info["num_units"]
        assert info["split_k"] <= info["k_blocks"]
        assert info["smem_bytes"] <= 232448
        assert info["tmem_cols"] in (128, 256, 512) and info["tmem_cols"] >= 2 * info["block_n"]
        assert info["pack_a"] == 0 and info["pack_b"] == 0 or w.name == "ragged_4097x4095x4100" \
            or w.name == "ragged_197x131x77"


def test_plan_ragged_workload_packs_and_uses_plain_stores(lib):
    """4097 x 4095 x 4100: lda = 4100 bf16 (8200 B) and ldb = 4095 (8190 B)
    are not 16-byte multiples, so both operands are packed; ldc = 4095 fp32
    (16380 B) rules out TMA stores of C."""
    w = synth.WORKLOADS["ragged_4097x4095x4100"]
    info = _plan(w)
    assert info["pack_a"] == 1 and info["pack_b"] == 1 and info["epilogue"] == 2
    assert info["tiles_m"] == -(-4097 // info["block_m"]) and info["k_blocks"] == 65
    assert info["workspace_bytes"] >= 2 * (4097 * 4104 + 4100 * 4096)


def test_plan_split_k_workspace(lib):
    info = tg.plan(64, 2048, 8192, sm_count=152, options=tg.make_options(block_n=256, split_k=4))
    assert info["split_k"] == 4 and info["num_units"] == 8 * 4
    assert info["workspace_bytes"] >= 8 * 4 * 128 * 256 * 4


@pytest.mark.parametrize("opt", [dict(block_n=96), dict(block_n=256, stages=5), dict(split_k=10 ** 6),
                                 dict(epilogue=3), dict(max_ctas=-1), dict(cta_pair=3),
                                 dict(cta_pair=2, block_n=64), dict(cta_pair=2, block_n=128, stages=6)])
def test_plan_rejects_bad_overrides(lib, opt):
    with pytest.raises(tg.TgError):
        tg.plan(512, 512, 512, sm_count=152, options=tg.make_options(**opt))


def test_plan_rejects_tma_store_on_misaligned_c(lib):
    with pytest.raises(tg.TgError):
        tg.plan(64, 63, 64, ldc=63, sm_count=152, options=tg.make_options(epilogue=1))


def test_plan_pair_choices(lib):
    """Two-SM tiles for the large tensor-bound square problem; one CTA per
    tile where 256-row tiles would waste rows or leave pairs idle."""
    sq = _plan(synth.WORKLOADS["square_4096"])
    assert sq["cta_pair"] == 2 and sq["block_m"] == 256 and sq["block_n"] == 256
    assert sq["grid"] == 152 and sq["tiles_m"] == 16
    # 256 tiles on 76 pairs: 3 whole waves, the last 28 tiles shared (stream-K)
    assert sq["stream_k"] == 2 and sq["sk_tiles"] == 256 - 3 * 76
    sk = _plan(synth.WORKLOADS["skinny_64x28672x8192"])
    assert sk["cta_pair"] == 1
    forced = tg.plan(1000, 1000, 1000, sm_count=152, options=tg.make_options(cta_pair=2, block_n=128))
    assert forced["cta_pair"] == 2 and forced["block_m"] == 256 and forced["tiles_m"] == 4
    with pytest.raises(tg.TgError):
        tg.plan(1000, 1000, 1000, sm_count=152, options=tg.make_options(cta_pair=2, block_n=192))


def test_stream_k_schedule_covers_every_k_block_once(lib):
    """Host-side model of the stream-K schedule the kernel walks: whole
    tiles for the full waves, then contiguous k-block ranges; every (tile,
    k-block) is covered exactly once and parts are numbered in k order."""
    def owner(x, W, L):
        return min(W - 1, ((x + 1) * W - 1) // L)

    for tiles, kb, W in [(256, 64, 76), (64, 32, 7), (10, 1, 7), (5, 3, 16), (29, 65, 4), (96, 64, 76),
                         (176, 64, 76), (272, 65, 76), (1024, 128, 76), (80, 3, 76)]:
        if tiles % W == 0:
            continue
        dp = tiles // W
        sk_tiles = tiles - dp * W
        L = sk_tiles * kb
        # the shared tiles cut into P >= 2 equal parts when they fit, else
        # an even split over all workers
        P = min(W // sk_tiles, kb)
        SW = P * sk_tiles if P >= 2 else W
        cover, units = {}, {}
        for w in range(W):
            for i in range(dp):
                t = w + i * W
                for k in range(kb):
                    cover[(t, k)] = cover.get((t, k), 0) + 1
            pos, end = (w * L // SW, (w + 1) * L // SW) if w < SW else (0, 0)
            while pos < end:
                ts = pos // kb
                e = min(end, (ts + 1) * kb)
                first, last = owner(ts * kb, SW, L), owner((ts + 1) * kb - 1, SW, L)
                assert first <= w <= last
                units[w] = units.get(w, 0) + 1
                for k in range(pos - ts * kb, e - ts * kb):
                    cover[(dp * W + ts, k)] = cover.get((dp * W + ts, k), 0) + 1
                pos = e
        assert len(cover) == tiles * kb and set(cover.values()) == {1}
        if P >= 2:
            assert set(units.values()) == {1}  # no range crosses a tile
        if tiles > W:  # (with fewer tiles than SMs the grid shrinks to the tiles)
            p = tg.plan(128 * tiles, 64, 64 * kb, sm_count=W,
                        options=tg.make_options(block_n=64, cta_pair=1, stream_k=2))
            assert p["sk_tiles"] == sk_tiles


def test_plan_stream_k_overrides(lib):
    off = tg.plan(4096, 4096, 4096, sm_count=152, options=tg.make_options(stream_k=1))
    assert off["stream_k"] == 1 and off["sk_tiles"] == 0
    with pytest.raises(tg.TgError):
        tg.plan(4096, 4096, 4096, sm_count=152, options=tg.make_options(stream_k=2, split_k=2))
    full = tg.plan(4096, 4096, 4096, sm_count=152,
                   options=tg.make_options(stream_k=2, cta_pair=2, max_ctas=128))
    # 256 tiles on 64 pairs: the last wave is full, nothing to balance
    assert full["stream_k"] == 1


def test_plan_honours_overrides(lib):
    info = tg.plan(1000, 1000, 1000, sm_count=152,
                   options=tg.make_options(block_n=192, stages=3, split_k=2, max_ctas=5, force_pack=1))
    assert (info["block_n"], info["stages"], info["split_k"], info["grid"]) == (192, 3, 2, 5)
    assert info["pack_a"] == 1 and info["pack_b"] == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """No CPU fallback: a missing library is an error, not a slower path."""
    monkeypatch.setattr(_abi, "_LIB", None)
    monkeypatch.setattr(_abi, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _abi.load()


def test_tune_rejects_bad_arguments_before_any_cuda_call(lib):
    best = tg.tg_options()
    us = ctypes.c_float(0)
    good = (1 << 30, 1 << 36, 1 << 40, 64, 64, 64, 64, 64, 64, 1, 0, 0, 0)
    assert tg.tg_tune(*good, None, None, 0, best, us) == tg.TG_ERR_INVALID_ARG      # reps < 1
    assert tg.tg_tune(*good, None, None, 101, best, us) == tg.TG_ERR_INVALID_ARG    # reps > 100
    assert tg.tg_tune(*good, None, None, 3, None, us) == tg.TG_ERR_INVALID_ARG      # no output
    bad = (1 << 30, 1 << 36, 1 << 40, 64, 64, 64, 32, 64, 64, 1, 0, 0, 0)           # lda < K
    assert tg.tg_tune(*bad, None, None, 3, best, us) == tg.TG_ERR_INVALID_ARG
    # empty problem: nothing to time, the base options come back
    empty = (1 << 30, 1 << 36, 1 << 40, 0, 64, 64, 64, 64, 64, 1, 0, 0, 0)
    base = tg.make_options(a_col_major=0, stages=4)
    assert tg.tg_tune(*empty, None, base, 3, best, us) == tg.TG_OK
    assert best.stages == 4 and us.value == 0.0


def test_mxfp8_rejects_bad_arguments_before_any_cuda_call(lib):
    """Block-scaled entry: scale pointers, pitches, strides, options and
    overlaps are checked on the host (fake device addresses, no GPU)."""
    M, N, K = 256, 256, 256
    A, B, D = 0x100000, 0x200000, 0x300000
    SF = 0x400000

    def call(sfa=SF, ld_sfa=8, s_sfa=0, sfb=SF, ld_sfb=8, s_sfb=0, opt=None, batch=1, sA=0, sB=0,
             fa=0, K=K):
        return tg.tg_gemm_mxfp8(A, B, D, M, N, K, K, K, N, batch, sA, sB, M * N, fa, 0,
                                sfa, ld_sfa, s_sfa, sfb, ld_sfb, s_sfb, None, None, opt)

    bad = tg.TG_ERR_INVALID_ARG
    assert call(sfa=None) == bad
    assert call(sfb=None) == bad
    assert call(ld_sfa=7) == bad                        # < ceil(K/32)
    assert call(ld_sfb=7) == bad
    assert call(s_sfa=-8) == bad
    assert call(fa=2) == bad                            # unknown format
    assert call(opt=tg.make_options(block_n=256)) == bad
    assert call(opt=tg.make_options(block_n=64)) == bad
    assert call(opt=tg.make_options(cta_pair=2)) == bad
    assert call(opt=tg.make_options(stages=6)) == bad
    assert call(opt=tg.make_options(a_col_major=1)) == bad
    # A shared across the batch but its scales not
    assert call(batch=2, sA=0, sB=N * K, s_sfa=M * 8) == bad
    # scales overlapping D
    assert call(sfa=D + 64) == bad
    # valid calls get past every host check (and then need a GPU): both tile
    # widths plan, with and without options
    assert call() == tg.TG_ERR_CUDA
    for bn in (128, 192, 224):
        for st in (2, 4):
            assert call(opt=tg.make_options(block_n=bn, stages=st)) == tg.TG_ERR_CUDA
    assert call(opt=tg.make_options(split_k=2)) == tg.TG_ERR_CUDA
    # the default width for a wide N (224 columns) plans too
    wide = tg.tg_gemm_mxfp8(A, B, 0x10000000, M, 4096, K, K, K, 4096, 1, 0, 0, 0, 0, 0,
                            0x20000000, 8, 0, 0x30000000, 8, 0, None, None, None)
    assert wide == tg.TG_ERR_CUDA
    assert call(opt=tg.make_options(stream_k=2)) == tg.TG_ERR_CUDA
    # K == 0: no scales needed, nothing to check (and M == 0: nothing to do)
    assert tg.tg_gemm_mxfp8(A, B, D, 0, N, K, K, K, N, 1, 0, 0, 0, 0, 0,
                            SF, 8, 0, SF, 8, 0, None, None, None) == tg.TG_OK


def test_plan_8bit_and_block_scaled_choices(lib):
    """tg_plan with opt->operands: the 8-bit planner's measured choices
    (two-SM 256-wide tiles for long K and a full wave, one CTA otherwise,
    192 wide on the skinny shape, stream-K only with the shared tiles cut
    into parts and 32 k-blocks or more) and the
    block-scaled widths (224 where tensor memory allows, 192 on the skinny
    shape), host-only."""
    p = tg.plan(4096, 4096, 4096, sm_count=152, operands="fp8")
    # stream-K with the 28 shared tiles cut in two (32 k-blocks of 128)
    assert (p["block_n"], p["cta_pair"], p["stream_k"], p["block_k"], p["sk_tiles"]) == (256, 2, 2, 128, 28)
    assert tg.plan(4096, 4096, 2048, sm_count=152, operands="fp8")["stream_k"] == 1  # 16 k-blocks
    assert tg.plan(8192, 8192, 8192, sm_count=152, operands="fp8")["cta_pair"] == 2
    assert tg.plan(4096, 4096, 1024, sm_count=152, operands="fp8")["cta_pair"] == 1   # short K
    assert tg.plan(2048, 2048, 2048, sm_count=152, operands="fp8")["cta_pair"] == 1   # under a wave
    # ... unless asked for
    assert tg.plan(16, 16, 16, sm_count=152, operands="fp8",
                   options=tg.make_options(block_n=256, cta_pair=2))["cta_pair"] == 2
    assert tg.plan(64, 28672, 8192, sm_count=152, operands="fp8")["block_n"] == 192
    p = tg.plan(4096, 4096, 4096, sm_count=152, operands="mxfp8")
    assert (p["block_n"], p["cta_pair"], p["tmem_cols"]) == (224, 1, 512)
    # the re-arranged scales: 512 bytes per 128 rows of A / per 128 columns
    # of a B tile (two blocks for 224) per k-block of 128
    assert p["workspace_bytes"] == 32 * 32 * 512 + 19 * 32 * 2 * 512
    assert tg.plan(64, 28672, 8192, sm_count=152, operands="mxfp8")["block_n"] == 192
    assert tg.plan(4096, 4096, 4096, sm_count=152, operands="mxfp8",
                   options=tg.make_options(block_n=128))["block_n"] == 128


def test_plan_8bit_rejections(lib):
    def plan(M, N, K, ops, **kw):
        o = tg.make_options(**kw)
        o.operands = tg.OPERAND_FAMILIES[ops] if ops in tg.OPERAND_FAMILIES else ops
        return tg.tg_plan(0x1000, 0x100000000, 0x200000000, M, N, K, K, K, N, 1, 0, 0, 0, 152, o)[0]

    assert plan(256, 256, 256, "mxfp8", block_n=256) == tg.TG_ERR_INVALID_ARG
    assert plan(256, 256, 256, "mxfp8", cta_pair=2) == tg.TG_ERR_INVALID_ARG
    assert plan(256, 256, 256, "fp8", a_col_major=1) == tg.TG_ERR_INVALID_ARG
    assert plan(256, 256, 256, 4) == tg.TG_ERR_INVALID_ARG
    assert plan(256, 256, 264, "fp8") == tg.TG_ERR_UNSUPPORTED  # rows of 264 bytes: not 16-byte multiples
    assert plan(256, 256, 256, "fp8") == tg.TG_OK
    # packed 4-bit: K and pitches count elements, two a byte
    assert plan(256, 256, 255, "mxfp4") == tg.TG_ERR_INVALID_ARG  # half a byte
    assert plan(256, 256, 272, "mxfp4") == tg.TG_ERR_UNSUPPORTED  # rows of 136 bytes
    assert plan(256, 256, 256, "mxfp4", block_n=224, stages=4) == tg.TG_ERR_INVALID_ARG
    assert plan(256, 256, 256, "mxfp4", block_n=256) == tg.TG_ERR_INVALID_ARG
    assert plan(256, 256, 256, "mxfp4") == tg.TG_OK


def test_plan_4bit_block_scaled(lib):
    """The packed 4-bit family: 256 elements of K per k-block (128 bytes a
    row), one-CTA tiles of 128, 192 or 224 columns, 224 with a two-slot
    ring; the scale scratch holds two blocks per 128 rows and k-block."""
    p = tg.plan(4096, 4096, 4096, sm_count=152, operands="mxfp4")
    assert p["block_k"] == 256 and p["k_blocks"] == 16 and p["cta_pair"] == 1
    # the two-slot 224-wide tiles only on request (measured slower)
    assert p["block_n"] in (128, 192) and p["stages"] == 4
    q = tg.plan(4096, 4096, 4096, sm_count=152, operands="mxfp4", options=tg.make_options(block_n=224))
    assert (q["block_n"], q["stages"]) == (224, 2)
    for bn, st in ((128, 4), (192, 4), (224, 2), (128, 2)):
        q = tg.plan(1000, 1000, 1056, sm_count=152, operands="mxfp4",
                    options=tg.make_options(block_n=bn, stages=st))
        assert (q["block_n"], q["stages"]) == (bn, st)
        tiles_m, tiles_n, kb = -(-1000 // 128), -(-1000 // bn), -(-1056 // 256)
        scales = -(-tiles_m * kb * 1024 // 256) * 256 + -(-tiles_n * kb * 1024 * -(-bn // 128) // 256) * 256
        assert q["workspace_bytes"] == scales


def test_c_caller_links_and_plans(lib):
    """A plain C program (no Python, no torch) includes the header, links the
    library and uses it host-only: plan queries for the three operand
    families, argument rejection and status strings."""
    from tiled_gemm_codegen_gb300 import build as _build

    src = r"""
#include <stdio.h>
#include <string.h>
#include "tg_gemm.h"
int main(void) {
  tg_plan_info info;
  tg_options opt;
  memset(&opt, 0, sizeof(opt));
  const void *A = (const void *)0x1000, *B = (const void *)0x100000000ull;
  const float *C = (const float *)0x200000000ull;
  if (tg_plan(A, B, C, 4096, 4096, 4096, 4096, 4096, 4096, 1, 0, 0, 0, 152, &opt, &info) != TG_OK) return 1;
  printf("%d %d %d %d\n", info.block_n, info.cta_pair, info.stages, info.k_blocks);
  opt.operands = 2;  /* block-scaled 8-bit: B stored N x K */
  if (tg_plan(A, B, C, 4096, 4096, 4096, 4096, 4096, 4096, 1, 0, 0, 0, 152, &opt, &info) != TG_OK) return 2;
  printf("%d %d %d %d\n", info.block_n, info.cta_pair, info.stages, info.k_blocks);
  /* lda < K is rejected before anything else happens */
  tg_status st = tg_gemm(A, B, (float *)C, 64, 64, 64, 32, 64, 64, 1, 0, 0, 0, NULL);
  printf("%d %s\n", (int)st, tg_status_string(st));
  return 0;
}
"""
    libpath = _build.library_path()
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "caller.c")
        exe = os.path.join(d, "caller")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe, libpath,
                        "-Wl,-rpath," + os.path.dirname(libpath)], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0].split() == ["256", "2", "6", "64"]       # bf16: two-SM 256 x 256 tiles, 64-element k-blocks
    assert out[1].split() == ["224", "1", "4", "32"]       # MXFP8: 224-wide tiles, 128-element k-blocks
    assert out[2].split()[0] == str(tg.TG_ERR_INVALID_ARG)


def test_checks_build_loads_and_plans_host_only():
    """The TG_DEBUG_CHECKS build exports every entry point the product build
    does and plans without a GPU like it."""
    chk = tg.load_checks()
    lib = tg.load()
    info_a, info_b = tg._abi.tg_plan_info(), tg._abi.tg_plan_info()
    for L, info in ((lib, info_a), (chk, info_b)):
        assert L.tg_plan(0x1000, 0x100000000, 0x200000000, 4096, 4096, 4096, 4096, 4096, 4096, 1, 0, 0, 0, 152,
                         None, ctypes.byref(info)) == tg.TG_OK
    assert info_a.as_dict() == info_b.as_dict()
    assert chk.tg_status_string(tg.TG_ERR_DEVICE_CHECK) == b"device-side consistency check failed"


def test_plan_rules_from_the_tuner_sweep():
    """The planner's measured rules (default plan against the run-time
    tuner's best on GB300): no stream-K with short partial units, no two-SM tiles
    when their rows would be half padding or a tile has few k-blocks, no
    tile twice as wide as N - and the five workloads keep their plans."""
    def P(M, N, K, b=1):
        return tg.plan(M, N, K, b, sm_count=152)
    assert P(2048, 8192, 2048)["stream_k"] == 2          # 32 k-blocks, shared tiles in halves
    assert P(4096, 1536, 2048)["stream_k"] == 1          # in thirds: parts of 10 k-blocks
    assert P(4096, 4096, 4096)["stream_k"] == 2          # 64 k-blocks
    assert P(128, 4096, 4096)["cta_pair"] == 1           # M = 128
    assert P(512, 512, 512, 32)["cta_pair"] == 1         # 8 k-blocks a tile
    assert P(4096, 128, 4096)["block_n"] <= 128          # N = 128
    p = P(4096, 4096, 4096)
    assert (p["block_n"], p["cta_pair"], p["stages"]) == (256, 2, 6)
    p = P(4097, 4095, 4100)
    assert (p["block_n"], p["cta_pair"], p["stream_k"]) == (256, 2, 2)
    p = P(384, 640, 1000, 64)
    assert (p["block_n"], p["cta_pair"], p["stages"]) == (256, 1, 4)
    p = P(64, 28672, 8192)
    assert (p["block_n"], p["cta_pair"]) == (192, 1)
    # the rules shape the planner's own choices only: a requested form is
    # always planned (two-SM tiles for a 39-column output, stream-K with
    # few k-blocks)
    q = tg.plan(693, 39, 719, 2, sm_count=152, options=tg.make_options(cta_pair=2))
    assert q["cta_pair"] == 2
    q = tg.plan(2048, 8192, 2048, sm_count=152, options=tg.make_options(stream_k=2))
    assert q["stream_k"] == 2


def test_plan_rules_for_every_operand_family():
    """The narrowest width that holds N, no two-SM tile that spans all of N,
    and (8-bit) no two-SM tile with fewer than 20 k-blocks; every operand
    family still has a plan for every narrow N, and a requested width is
    kept."""
    for ops in ("bf16", "fp8", "mxfp8", "mxfp4"):
        for N in list(range(1, 300, 7)) + [64, 128, 192, 256]:
            p = tg.plan(4096, N, 4096, sm_count=152, operands=ops)
            assert p["block_n"] >= 64 and p["grid"] > 0, (ops, N)
            if N <= 128:
                assert p["block_n"] <= 128, (ops, N, p["block_n"])
            if N <= p["block_n"]:
                assert p["cta_pair"] == 1, (ops, N)
        assert tg.plan(4096, 128, 4096, sm_count=152, operands=ops,
                       options=tg.make_options(block_n=192))["block_n"] == 192
    for b, M, N, K in ((1, 16384, 16384, 512), (32, 512, 512, 512), (1, 2048, 8192, 2048)):
        assert tg.plan(M, N, K, b, sm_count=152, operands="fp8")["cta_pair"] == 1
    p = tg.plan(4096, 4096, 4096, sm_count=152, operands="fp8")
    assert (p["block_n"], p["cta_pair"]) == (256, 2)                 # 32 k-blocks
    assert tg.plan(4096, 160, 4096, sm_count=152)["cta_pair"] == 1
    assert tg.plan(4096, 160, 4096, sm_count=152, options=tg.make_options(cta_pair=2))["cta_pair"] == 2


def test_plan_half_height_a_rings():
    """Outputs of at most 64 rows take 64-row A slots (8 at width 128, 6 at
    width 192) when the ring depth is the planner's or that one; an explicit
    other depth, two-SM tiles, widths without such an instance and outputs
    of more than 64 rows keep the 128-row slots."""
    def P(M, N=4096, K=4096, ops="bf16", **kw):
        return tg.plan(M, N, K, sm_count=152, operands=ops, options=tg.make_options(**kw) if kw else None)
    for ops in ("bf16", "fp8"):
        for bn, s in ((128, 8), (192, 6)):
            for M in (1, 33, 64):
                p = P(M, ops=ops, block_n=bn)
                assert (p["block_m"], p["stages"]) == (64, s), (ops, bn, M, p)
                p = P(M, ops=ops, block_n=bn, stages=s)
                assert p["block_m"] == 64
                p = P(M, ops=ops, block_n=bn, stages=4)
                assert (p["block_m"], p["stages"]) == (128, 4)
            assert P(65, ops=ops, block_n=bn)["block_m"] == 128
        assert P(64, ops=ops, block_n=256)["block_m"] == 128
    assert P(64, block_n=64)["block_m"] == 128
    assert P(64, block_n=128, cta_pair=2)["block_m"] == 256
    # block-scaled operands keep their own rings
    assert P(64, ops="mxfp8")["block_m"] == 128


def test_direct_plan_fields_and_requests(lib):
    """direct = 2 asks for the direct-load kernel: bf16 operands and no
    override but the operand layouts; any other override with it is an
    invalid request."""
    d = tg.make_options(direct=2)
    info = tg.plan(300, 200, 600, 3, sm_count=152, options=d)
    assert info["direct"] == 2 and (info["block_m"], info["block_n"]) == (128, 64)
    assert (info["tiles_m"], info["tiles_n"], info["k_blocks"]) == (3, 4, 10)
    assert info["grid"] == info["num_units"] == 3 * 3 * 4 and info["stages"] == 4
    assert info["tmem_cols"] == 64 and info["workspace_bytes"] == 0 and info["epilogue"] == 2
    assert tg.plan(5, 5, 40, sm_count=152, options=d)["stages"] == 1
    for extra in (dict(block_n=128), dict(stages=4), dict(split_k=2), dict(force_pack=1), dict(epilogue=1),
                  dict(cta_pair=2), dict(stream_k=2), dict(max_ctas=8)):
        with pytest.raises(tg.TgError):
            tg.plan(300, 200, 600, sm_count=152, options=tg.make_options(direct=2, **extra))
    with pytest.raises(tg.TgError):
        tg.plan(300, 200, 600, sm_count=152, options=tg.make_options(direct=3))
    with pytest.raises(tg.TgError):  # 8-bit operands
        tg.plan(256, 256, 256, sm_count=152, operands="fp8", options=tg.make_options(direct=2))
    # overrides the direct kernel shares are accepted
    assert tg.plan(300, 200, 600, sm_count=152, options=tg.make_options(direct=2, block_n=64, split_k=1, cta_pair=1,
                                                                      stream_k=1, epilogue=2))["direct"] == 2


def test_direct_planner_rule(lib):
    """The planner's own choice: at most one tile per SM, and at most 8
    k-blocks when both operands can be staged in 16-byte units (aligned,
    contiguous extent a multiple of 8), 5 when one needs the persistent
    kernel's realign pass (staged element by element), else 2."""
    def direct(M, N, K, batch=1, lda=None, ldb=None, opts=None):
        return tg.plan(M, N, K, batch, sm_count=152, lda=lda, ldb=ldb, options=opts)["direct"] == 2
    assert direct(197, 131, 77)                    # odd pitches, 2 k-blocks
    assert direct(129, 65, 257)                    # odd pitch, 5 k-blocks
    assert not direct(100, 300, 500, lda=501)      # 8 k-blocks
    assert direct(1000, 1000, 64)                  # 128 tiles, 1 k-block
    assert direct(128, 128, 128)
    assert direct(256, 256, 256) and direct(512, 512, 512)      # 16-byte units, 4 and 8 k-blocks
    assert not direct(128, 128, 1024)              # 16 k-blocks
    assert not direct(256, 256, 260, lda=264)      # aligned but K not a multiple of 8: 5 k-blocks > 2
    assert direct(256, 250, 128, ldb=256)          # aligned, N not a multiple of 8: 2 k-blocks
    assert not direct(4096, 4096, 64)              # 2048 tiles
    assert not direct(2048, 2048, 128)             # 512 tiles
    assert direct(64, 64, 64, 64)                  # 64 problems of one tile
    assert not direct(128, 128, 128, opts=tg.make_options(block_n=64))  # an override: the persistent kernel
    assert not direct(128, 128, 128, opts=tg.make_options(direct=1))
    assert not direct(4096, 4096, 4096)


def test_plan_invariants_on_random_calls(lib):
    """Random extents, batches, pointer alignments, layouts and overrides
    (some invalid): the planner either refuses with TG_ERR_INVALID_ARG /
    TG_ERR_UNSUPPORTED or returns a plan whose fields are consistent - tile
    counts cover the problem, the grid and the resources fit one GB300, and
    the direct-load kernel's plans have its fixed geometry."""
    import random

    r = random.Random(2024)
    SMEM_MAX, SMS = 232448, 152
    for case in range(1500):
        M = int(2 ** r.uniform(0, 14))
        N = int(2 ** r.uniform(0, 14))
        K = int(2 ** r.uniform(0, 14))
        batch = r.choice([1, 1, 1, 2, 7, 64])
        a_cm, b_cm = r.random() < 0.25, r.random() < 0.25
        a_rows, a_cols = (K, M) if a_cm else (M, K)
        b_rows, b_cols = (N, K) if b_cm else (K, N)
        lda = a_cols + r.choice([0, 0, 1, 8])
        ldb = b_cols + r.choice([0, 0, 3, 8])
        opts = dict(a_col_major=int(a_cm), b_col_major=int(b_cm))
        pick = r.random()
        if pick < 0.15:
            opts["direct"] = r.choice([1, 2])
        elif pick < 0.3:
            opts["block_n"] = r.choice([64, 128, 192, 256])
        elif pick < 0.4:
            opts["split_k"] = r.choice([1, 2, 3])
        elif pick < 0.5:
            opts["stream_k"] = r.choice([1, 2])
        elif pick < 0.55:
            opts["cta_pair"] = r.choice([1, 2])
        A = 0x1000 + 2 * r.choice([0, 0, 1, 4])
        try:
            info = tg.plan(M, N, K, batch, lda=lda, ldb=ldb, strideA=a_rows * lda, strideB=b_rows * ldb,
                           A=A, sm_count=SMS, options=tg.make_options(**opts))
        except tg.TgError as e:
            assert e.status in (tg.TG_ERR_INVALID_ARG, tg.TG_ERR_UNSUPPORTED), (case, e.status)
            continue
        kb = -(-K // 64)
        where = (case, M, N, K, batch, opts, info)
        assert info["k_blocks"] == kb and info["smem_bytes"] <= SMEM_MAX, where
        assert info["tiles_m"] == -(-M // (128 * info["cta_pair"])) or info["block_m"] == 64, where
        assert info["tiles_n"] == -(-N // info["block_n"]), where
        if info["direct"] == 2:
            assert opts.get("direct", 0) != 1, where
            assert (info["block_m"], info["block_n"], info["cta_pair"], info["split_k"]) == (128, 64, 1, 1), where
            assert info["grid"] == info["num_units"] == batch * info["tiles_m"] * info["tiles_n"], where
            assert info["stages"] == min(4, kb) and info["tmem_cols"] == 64, where
            assert info["pack_a"] == info["pack_b"] == 0 and info["workspace_bytes"] == 0, where
            if opts.get("direct", 0) == 0:
                assert info["num_units"] <= SMS and kb <= 8, where
        else:
            assert info["direct"] == 1 and opts.get("direct", 0) != 2, where
            assert info["num_units"] == batch * info["tiles_m"] * info["tiles_n"] * info["split_k"], where
            assert 1 <= info["grid"] <= SMS and info["grid"] <= info["num_units"] * info["cta_pair"], where
            assert info["cta_pair"] == 1 or info["grid"] % 2 == 0, where
            assert 1 <= info["split_k"] <= kb and 2 <= info["stages"] <= 8, where
            assert info["tmem_cols"] in (128, 256, 512) and info["tmem_cols"] >= 2 * info["block_n"], where
            assert info["stream_k"] == 1 or info["split_k"] == 1, where
