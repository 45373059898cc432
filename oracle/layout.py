"""TIRx layout calculus, restated from TVM "Tensor Layout" (docs/tirx/layout.rst).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* ``TileLayout`` - shard ``D`` / replica ``R`` / offset ``O`` with the
  four-step forward mapping of section "Forward mapping" (flatten, split,
  accumulate + offset, broadcast replicas).
* ``parse_layout`` - reads the pages' textual form, e.g.
  ``S[(8,2,4,2):(4@laneid,1@warpid,1@laneid,1)] + R[2:4@warpid] + 5@warpid``;
  a stride with no ``@axis`` lands on the default memory axis ``m``.
* ``swizzle_addr`` / ``swizzle_params`` - section "SwizzleLayout,
  ComposeLayout": ``addr(m) = f(m >> M) * 2^M + (m mod 2^M)`` with
  ``f(x) = x xor ((x & ((2^B - 1) << S)) >> S)``, and the parameter choice
  ``M = bitlen(128 / dtype_bits) - 1``, ``B`` = 1/2/3 for 32B/64B/128B, ``S = 3``.
* ``bank_line`` - section "Bank and line of an element":
  ``bankword = floor(a * b / 4)``, ``bank = bankword mod 32``,
  ``line = floor(bankword / 32)``.

Pinned by ``tests/test_layout.py`` against the page's printed tables
(tensor-core register tile, Blackwell tensor memory, 128B-swizzle worked
example) stored under ``tests/golden/``.
"""
from __future__ import annotations

import itertools
import re
from dataclasses import dataclass, field

DEFAULT_AXIS = "m"


@dataclass(frozen=True)
class Iter:
    extent: int
    stride: int
    axis: str


@dataclass
class TileLayout:
    shard: list[Iter]
    replica: list[Iter] = field(default_factory=list)
    offset: dict[str, int] = field(default_factory=dict)

    def size(self) -> int:
        n = 1
        for it in self.shard:
            n *= it.extent
        return n

    def admits(self, shape) -> bool:
        """A shape is admitted when its total size equals the product of the
        shard extents."""
        n = 1
        for s in shape:
            n *= s
        return n == self.size()

    def axes(self) -> list[str]:
        seen: list[str] = []
        for it in list(self.shard) + list(self.replica):
            if it.axis not in seen:
                seen.append(it.axis)
        for a in self.offset:
            if a not in seen:
                seen.append(a)
        return seen

    def evaluate(self, shape, x) -> list[dict[str, int]]:
        """L(x): the set of physical coordinates of logical index ``x``.

        Returned as a list of {axis: coordinate} dicts, one per replica
        combination (a singleton list when there is no replica)."""
        if len(shape) != len(x):
            raise ValueError("rank mismatch")
        if not self.admits(shape):
            raise ValueError(f"shape {shape} not admitted (size {self.size()})")
        for xd, sd in zip(x, shape):
            if not 0 <= xd < sd:
                raise ValueError(f"coordinate {x} outside shape {shape}")
        # 1. flatten row-major
        flat = 0
        for d, xd in enumerate(x):
            inner = 1
            for e in shape[d + 1:]:
                inner *= e
            flat += xd * inner
        # 2. split across shard extents (component k uses the product of the
        #    extents after it as its divisor)
        comps = []
        for k, it in enumerate(self.shard):
            inner = 1
            for later in self.shard[k + 1:]:
                inner *= later.extent
            comps.append((flat // inner) % it.extent)
        # 3. accumulate on axes, then add the offset
        base = {a: 0 for a in self.axes()}
        for c, it in zip(comps, self.shard):
            base[it.axis] += c * it.stride
        for a, o in self.offset.items():
            base[a] += o
        # 4. broadcast replicas
        out = []
        for r in itertools.product(*[range(it.extent) for it in self.replica]):
            coord = dict(base)
            for rt, it in zip(r, self.replica):
                coord[it.axis] += rt * it.stride
            out.append(coord)
        return out

    def components(self, shape, x) -> tuple[int, ...]:
        """The split components (c_0, ..., c_{n-1}) of step 2, for tables."""
        flat = 0
        for d, xd in enumerate(x):
            inner = 1
            for e in shape[d + 1:]:
                inner *= e
            flat += xd * inner
        comps = []
        for k, it in enumerate(self.shard):
            inner = 1
            for later in self.shard[k + 1:]:
                inner *= later.extent
            comps.append((flat // inner) % it.extent)
        return tuple(comps)


_TERM = re.compile(r"^\s*(-?\d+)\s*(?:@\s*([A-Za-z_][A-Za-z_0-9]*))?\s*$")


def _terms(text: str) -> list[tuple[int, str]]:
    out = []
    for part in text.split(","):
        m = _TERM.match(part)
        if not m:
            raise ValueError(f"bad term {part!r}")
        out.append((int(m.group(1)), m.group(2) or DEFAULT_AXIS))
    return out


def _ints(text: str) -> list[int]:
    return [int(p) for p in text.split(",")]


def parse_layout(text: str) -> TileLayout:
    """Parse ``S[(e..):(s@a..)] [+ R[(e..):(s@a..)] | R[e:s@a]] [+ n@axis ...]``."""
    s = text.strip()
    m = re.match(r"^S\[\(([^)]*)\):\(([^)]*)\)\]", s)
    if not m:
        raise ValueError("layout must start with a shard S[(...):(...)]")
    extents = _ints(m.group(1))
    strides = _terms(m.group(2))
    if len(extents) != len(strides):
        raise ValueError("shard extents and strides differ in length")
    shard = [Iter(e, st, ax) for e, (st, ax) in zip(extents, strides)]
    rest = s[m.end():]
    replica: list[Iter] = []
    offset: dict[str, int] = {}
    for piece in [p.strip() for p in rest.split("+") if p.strip()]:
        if piece.startswith("R["):
            body = piece[2:-1].strip()
            if body.startswith("("):
                mm = re.match(r"^\(([^)]*)\):\(([^)]*)\)$", body)
                if not mm:
                    raise ValueError(f"bad replica {piece!r}")
                ex = _ints(mm.group(1))
                st = _terms(mm.group(2))
            else:
                e_txt, s_txt = body.split(":", 1)
                ex = [int(e_txt)]
                st = _terms(s_txt)
            replica += [Iter(e, v, ax) for e, (v, ax) in zip(ex, st)]
        else:
            for v, ax in _terms(piece):
                offset[ax] = offset.get(ax, 0) + v
    return TileLayout(shard, replica, offset)


def bitlen(n: int) -> int:
    return int(n).bit_length()


def swizzle_params(dtype_bits: int, mode_bytes: int) -> tuple[int, int, int]:
    """(M, B, S) for a dtype width and a 32B/64B/128B swizzle mode."""
    B = {32: 1, 64: 2, 128: 3}[mode_bytes]
    M = bitlen(128 // dtype_bits) - 1
    return M, B, 3


def swizzle_addr(m: int, M: int, B: int, S: int) -> int:
    """The SwizzleLayout map of a linear element address ``m``."""
    if S < B:
        raise ValueError("well-formedness requires S >= B")
    x = m >> M
    mask = ((1 << B) - 1) << S
    f = x ^ ((x & mask) >> S)
    return f * (1 << M) + (m % (1 << M))


def bank_line(addr_elems: int, elem_bytes: int) -> tuple[int, int]:
    """(bank, line) of an element at element address ``addr_elems``."""
    bankword = (addr_elems * elem_bytes) // 4
    return bankword % 32, bankword // 32
