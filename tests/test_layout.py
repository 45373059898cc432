"""TIRx layout helpers against the layout page's printed tables (CPU only).

Pins: TVM "Tensor Layout" - the tensor-core register tile table, the
Blackwell tensor-memory table and the 128B-swizzle worked example, stored as
fixtures in ``tests/golden/``.  Then two design checks on the library's
shared-memory use, made with the same page formulas.
"""
from __future__ import annotations

import os

import pytest

from oracle import layout

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(name):
    meta, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line and line.split(":", 1)[0] in ("layout", "shape", "params"):
                k, v = line.split(":", 1)
                meta[k] = v.strip()
            else:
                rows.append(line.split())
    return meta, rows


def test_register_tile_table():
    meta, rows = _read("tirx_register_tile.txt")
    lay = layout.parse_layout(meta["layout"])
    shape = tuple(int(s) for s in meta["shape"].split())
    assert len(rows) == 6
    for r in rows:
        i, j, flat = int(r[0]), int(r[1]), int(r[2])
        comps = tuple(int(x) for x in r[3:7])
        lane, warps, m = int(r[7]), {int(w) for w in r[8].split(",")}, int(r[9])
        assert 16 * i + j == flat
        assert lay.components(shape, (i, j)) == comps
        coords = lay.evaluate(shape, (i, j))
        assert {c["warpid"] for c in coords} == warps
        assert all(c["laneid"] == lane and c["m"] == m for c in coords)


def test_register_tile_closed_form():
    """The page's closed form: laneid = 4i + floor(j/2) mod 4,
    warpid = floor(j/8) + 5 + 4r, m = j mod 2, for every element."""
    meta, _ = _read("tirx_register_tile.txt")
    lay = layout.parse_layout(meta["layout"])
    for i in range(8):
        for j in range(16):
            coords = lay.evaluate((8, 16), (i, j))
            assert sorted(c["warpid"] for c in coords) == [j // 8 + 5, j // 8 + 9]
            for c in coords:
                assert c["laneid"] == 4 * i + (j // 2) % 4
                assert c["m"] == j % 2


def test_tensor_memory_table():
    meta, rows = _read("tirx_tensor_memory.txt")
    lay = layout.parse_layout(meta["layout"])
    shape = tuple(int(s) for s in meta["shape"].split())
    for r in rows:
        a, l, c, tl, tc = (int(x) for x in r)
        (coord,) = lay.evaluate(shape, (a, l, c))
        assert coord["TLane"] == tl and coord["TCol"] == tc
    # whole-tile: a bijection onto 128 lanes x 224 columns
    seen = set()
    for a in range(2):
        for l in range(0, 128, 7):
            for c in range(112):
                (coord,) = lay.evaluate(shape, (a, l, c))
                assert coord["TLane"] == l and coord["TCol"] == 112 * a + c
                seen.add((coord["TLane"], coord["TCol"]))
    assert max(tc for _, tc in seen) == 223


def test_accumulator_placement_of_the_library():
    """The library keeps a double-buffered BM x BN fp32 accumulator in tensor
    memory as S[(2,128,BN):(BN@TCol,1@TLane,1@TCol)] - the page's TMEM
    placement with BN columns per buffer.  For every tile width the library
    instantiates, both buffers fit the 512 columns of one SM."""
    for bn in (64, 128, 192, 256):
        lay = layout.parse_layout(f"S[(2,128,{bn}):({bn}@TCol,1@TLane,1@TCol)]")
        (last,) = lay.evaluate((2, 128, bn), (1, 127, bn - 1))
        assert last["TLane"] == 127 and last["TCol"] == 2 * bn - 1 < 512


def test_swizzle_parameters_from_dtype():
    assert layout.swizzle_params(16, 128) == (3, 3, 3)
    assert layout.swizzle_params(32, 128) == (2, 3, 3)
    assert layout.swizzle_params(8, 64) == (4, 2, 3)
    assert layout.swizzle_params(16, 32) == (3, 1, 3)


def test_swizzle_worked_example():
    meta, rows = _read("tirx_swizzle_128b_fp16.txt")
    bits, mode, M, B, S = (int(x) for x in meta["params"].split())
    assert layout.swizzle_params(bits, mode) == (M, B, S)
    for r in rows:
        i, addr, bank_sw, bank_plain = (int(x) for x in r)
        a = layout.swizzle_addr(64 * i + 0, M, B, S)
        assert a == addr
        assert layout.bank_line(a, 2)[0] == bank_sw
        assert layout.bank_line(64 * i, 2)[0] == bank_plain
    # the printed closed form holds for every element of the (8, 64) tile
    for i in range(8):
        for j in range(64):
            assert layout.swizzle_addr(64 * i + j, M, B, S) == 64 * i + 8 * ((j // 8) ^ i) + j % 8


@pytest.mark.parametrize("mode", [32, 64, 128])
@pytest.mark.parametrize("bits", [8, 16, 32])
def test_any_16B_column_is_conflict_free(mode, bits):
    """The page's key claim: with swizzle, reading any 8 x 16B column of a
    tile whose rows span the swizzle width touches 32 distinct banks."""
    M, B, S = layout.swizzle_params(bits, mode)
    elem = bits // 8
    row_elems = mode // elem
    per16 = 16 // elem
    for chunk in range(mode // 16):
        banks = set()
        for i in range(8):
            for e in range(per16):
                m = i * row_elems + chunk * per16 + e
                a = layout.swizzle_addr(m, M, B, S)
                banks.add(layout.bank_line(a, elem)[0])
        assert len(banks) == 32


def test_swizzle_is_bijection():
    for (M, B, S) in [(3, 3, 3), (2, 3, 3), (3, 2, 3), (3, 1, 3)]:
        n = 1 << (M + B + S)
        assert sorted(layout.swizzle_addr(m, M, B, S) for m in range(n)) == list(range(n))


def test_epilogue_staging_pattern_is_conflict_free():
    """Design check of the library's epilogue: each warp stages a 32 x 32
    fp32 sub-tile with Swizzle(2,3,3) (fp32, 128B); lane t writes 16-byte
    chunk q of row t.  A 16-byte store is served in quarter-warp phases of 8
    lanes; within every phase the 8 stores cover 32 distinct banks."""
    M, B, S = layout.swizzle_params(32, 128)
    for q in range(8):
        for phase in range(4):
            banks = []
            for t in range(8 * phase, 8 * phase + 8):
                for e in range(4):
                    a = layout.swizzle_addr(t * 32 + 4 * q + e, M, B, S)
                    banks.append(layout.bank_line(a, 4)[0])
            assert len(set(banks)) == 32
    # the unswizzled layout would serialise the same phase 8-way
    for phase in range(4):
        banks = [layout.bank_line(t * 32, 4)[0] for t in range(8 * phase, 8 * phase + 8)]
        assert len(set(banks)) == 1


def test_parse_rejects_bad_layout():
    with pytest.raises(ValueError):
        layout.parse_layout("R[2:4@warpid]")
    lay = layout.parse_layout("S[(4,8):(8,1)]")
    with pytest.raises(ValueError):
        lay.evaluate((4, 4), (0, 0))
