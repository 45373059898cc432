"""Seeded synthetic inputs for the bf16 GEMM: shared by the tests, the
benchmark and the oracle's callers.

This module draws random numbers and rounds them to bf16; it holds none of
the GEMM's arithmetic, and neither the oracle nor the CUDA library imports
the other through it.

Recipe (the pages fix no generator, so this is the plainest reproducible one):
* ``torch.Generator('cpu').manual_seed(seed)``; A is drawn before B, each in
  one call over its full ``[batch, M, K]`` / ``[batch, K, N]`` shape.
* ``uniform``: ``rand * 2 - 1`` in fp32 (U[-1, 1)); ``normal``: ``randn``
  (N(0, 1)); ``normal002``: ``randn * 0.02`` (N(0, 0.02^2)).  Then a
  round-to-nearest-even cast to bf16 (after rounding, U[-1, 1) can hold 1.0).
* ``int``: integers drawn uniformly from ``[-mag, mag]``; with
  ``mag^2 * K < 2^24`` every partial sum of the product is an exact fp32
  integer, so any summation order gives the same bits.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    M: int
    N: int
    K: int
    dist: str
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.batch * self.M * self.N * self.K

    @property
    def bytes_moved(self) -> int:
        """A and B in bf16 plus C in fp32, each moved once."""
        return self.batch * (2 * self.M * self.K + 2 * self.K * self.N + 4 * self.M * self.N)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("ragged_197x131x77", 1, 197, 131, 77, "uniform", 0),
        Workload("square_4096", 1, 4096, 4096, 4096, "uniform", 1),
        Workload("ragged_4097x4095x4100", 1, 4097, 4095, 4100, "normal", 2),
        Workload("batched_64x384x640x1000", 64, 384, 640, 1000, "uniform", 3),
        Workload("skinny_64x28672x8192", 1, 64, 28672, 8192, "normal002", 4),
    )
}


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "normal002":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * 0.02
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(batch: int, M: int, N: int, K: int, dist: str, seed: int):
    """A [batch, M, K] and B [batch, K, N] as contiguous CPU bf16 tensors
    (the leading batch dim is dropped when ``batch == 1``)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    a = _draw(gen, (batch, M, K), dist).to(torch.bfloat16)
    b = _draw(gen, (batch, K, N), dist).to(torch.bfloat16)
    if batch == 1:
        a, b = a[0], b[0]
    return a.contiguous(), b.contiguous()


def workload_inputs(w: Workload):
    return make_inputs(w.batch, w.M, w.N, w.K, w.dist, w.seed)


def int_magnitude(K: int) -> int:
    """Largest integer magnitude (<= 16) with mag^2 * K < 2^24."""
    mag = 16
    while mag > 1 and mag * mag * max(K, 1) >= (1 << 24):
        mag -= 1
    return mag


def make_int_inputs(batch: int, M: int, N: int, K: int, seed: int, mag: int | None = None):
    """Small-integer-valued bf16 inputs (exact in fp32 under any sum order)."""
    mag = int_magnitude(K) if mag is None else mag
    gen = torch.Generator("cpu").manual_seed(seed)
    a = torch.randint(-mag, mag + 1, (batch, M, K), generator=gen, dtype=torch.int32)
    b = torch.randint(-mag, mag + 1, (batch, K, N), generator=gen, dtype=torch.int32)
    a = a.to(torch.bfloat16)
    b = b.to(torch.bfloat16)
    if batch == 1:
        a, b = a[0], b[0]
    return a.contiguous(), b.contiguous()


def sample_indices(batch: int, M: int, N: int, count: int, seed: int,
                   tile_m: int = 128, tile_n: int = 64):
    """Output positions to check one by one at full size: every corner, the
    first/last row and column of every tile edge near the fringe, and
    ``count`` uniformly drawn positions.  Returns (bi, ii, jj) int64 arrays."""
    rng = np.random.default_rng(seed)
    pts = set()
    rows = {0, M - 1, max(M - 2, 0)}
    cols = {0, N - 1, max(N - 2, 0)}
    for t in range(0, M, tile_m):
        rows.update({t, min(t + tile_m - 1, M - 1)})
    for t in range(0, N, tile_n):
        cols.update({t, min(t + tile_n - 1, N - 1)})
    rows = sorted(rows)
    cols = sorted(cols)
    batches = sorted({0, batch - 1, batch // 2})
    # edge structure: all (fringe row x sampled col) and (sampled row x fringe col)
    edge_r = [r for r in rows if r >= M - tile_m or r < tile_m] or rows
    edge_c = [c for c in cols if c >= N - tile_n or c < tile_n] or cols
    for b in batches:
        for r in edge_r:
            for c in cols[:: max(1, len(cols) // 16)]:
                pts.add((b, r, c))
        for c in edge_c:
            for r in rows[:: max(1, len(rows) // 16)]:
                pts.add((b, r, c))
    for _ in range(count):
        pts.add((int(rng.integers(batch)), int(rng.integers(M)), int(rng.integers(N))))
    arr = np.array(sorted(pts), dtype=np.int64).reshape(-1, 3)
    return arr[:, 0].copy(), arr[:, 1].copy(), arr[:, 2].copy()


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a CPU bf16 tensor, as numpy uint16."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bf16")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ 8-bit operands
FP8_DTYPES = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}  # format code -> torch dtype


def make_fp8_codes(shape, fmt: int, seed: int, kind: str = "int") -> torch.Tensor:
    """Seeded 8-bit floating-point codes (uint8) of format ``fmt`` (0 E4M3,
    1 E5M2).  ``int``: integers drawn uniformly from [-16, 16] (E4M3) or
    [-8, 8] (E5M2), every one of them exact in the format; ``finite``: codes
    drawn uniformly among the format's finite values; ``normal``: N(0, 1)
    draws cast to the format by PyTorch (round to nearest)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    dt = FP8_DTYPES[fmt]
    if kind == "int":
        mag = 16 if fmt == 0 else 8
        v = torch.randint(-mag, mag + 1, tuple(shape), generator=gen).to(torch.float32)
        return v.to(dt).view(torch.uint8)
    if kind == "finite":
        allc = torch.arange(256, dtype=torch.uint8)
        ok = allc[torch.isfinite(allc.view(dt).to(torch.float32))]
        idx = torch.randint(0, ok.numel(), tuple(shape), generator=gen)
        return ok[idx]
    if kind == "normal":
        return torch.randn(tuple(shape), generator=gen).to(dt).view(torch.uint8)
    raise ValueError(kind)


def make_e8m0_codes(shape, seed: int, lo: int = 124, hi: int = 130) -> torch.Tensor:
    """Seeded E8M0 scale codes (uint8) drawn uniformly from [lo, hi]; the
    default range is scales 2^-3 .. 2^3."""
    gen = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, tuple(shape), generator=gen).to(torch.uint8)


# ------------------------------------------------------------ packed 4-bit operands
def make_fp4_codes(shape, seed: int, lo: int = 0, hi: int = 15) -> torch.Tensor:
    """Seeded 4-bit E2M1 codes (uint8, one code per element, values lo..hi
    drawn uniformly; the default covers all 16 codes, every one finite)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, tuple(shape), generator=gen).to(torch.uint8)


def pack_fp4_codes(codes: torch.Tensor) -> torch.Tensor:
    """[.., K] codes (K even) -> [.., K/2] bytes, element 2i in the low
    nibble of byte i and element 2i + 1 in the high nibble: the storage of
    the library's packed 4-bit operands.  A layout step, no arithmetic."""
    if codes.shape[-1] % 2:
        raise ValueError("K must be even")
    c = codes.to(torch.uint8).reshape(*codes.shape[:-1], -1, 2)
    return (c[..., 0] | (c[..., 1] << 4)).contiguous()
