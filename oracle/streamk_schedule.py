"""Stream-K work decomposition, restated in plain Python (test oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: GitHub issue "Stream-k matmul implementation very slow mostly because
of if/else inside for loop" (triton tracker), final code version:

* wrapper ``_call``: the grid of output tiles, iterations per tile, how many
  tiles go to the Stream-K wave (``tiles % g``, plus ``g`` more when
  "two_tiles" is on and more than ``g`` whole tiles would remain), and the even
  split of the Stream-K iterations over ``g`` programs, the first
  ``remainder`` programs taking one extra iteration;
* ``first_wave``: a program's iteration range, cut at tile boundaries into
  segments (one tile and one k-range each);
* ``full_tiles``: the remaining tiles, one per program, numbered after the
  Stream-K tiles;
* ``swizzle_tile`` / ``linear_tile``: tile id -> (tile row, tile column), the
  grouped raster with GROUP_M rows per group, or plain row-major order.

Where the page leaves a step open, the reading is:

* owner of a split tile = the segment that holds k-iteration 0; the other
  segments of the tile are its peers, in ascending k (the page instead lets the
  segment holding the last iteration store and the others add atomically);
* a persistent program that finishes its Stream-K range goes on with whole
  tiles ``sk + pid, sk + pid + g, ...`` (the page launches them as a second
  grid); the set of whole tiles is the same;
* ``all_streamk``: every tile goes to the Stream-K wave (``sk = tiles``), the
  plain form of splitting the whole iteration space evenly over the programs.
"""
from __future__ import annotations

from dataclasses import dataclass, field


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class Schedule:
    M: int
    N: int
    K: int
    BM: int
    BN: int
    BK: int
    g: int                  # programs in the Stream-K wave (0: no Stream-K)
    two_tiles: bool = True
    group_m: int = 8        # 0 selects the linear raster
    all_streamk: bool = False
    tiles_m: int = field(init=False)
    tiles_n: int = field(init=False)
    tiles: int = field(init=False)
    ipt: int = field(init=False)             # iterations per tile
    sk_tiles: int = field(init=False)        # tiles done by the Stream-K wave
    dp_tiles: int = field(init=False)        # tiles done whole
    sk_iters: int = field(init=False)        # total Stream-K iterations
    iters_per_prog: int = field(init=False)  # even share of each program
    iters_rem: int = field(init=False)       # programs that take one more

    def __post_init__(self):
        self.tiles_m = cdiv(self.M, self.BM)
        self.tiles_n = cdiv(self.N, self.BN)
        self.tiles = self.tiles_m * self.tiles_n
        self.ipt = cdiv(self.K, self.BK)
        if self.g > 0:
            sk = self.tiles % self.g
            if self.two_tiles and self.tiles - sk > self.g:
                sk += self.g
            if self.all_streamk:
                sk = self.tiles
            self.sk_tiles = sk
            self.dp_tiles = self.tiles - sk
            self.sk_iters = sk * self.ipt
            self.iters_per_prog = self.sk_iters // self.g
            self.iters_rem = self.sk_iters % self.g
        else:
            self.sk_tiles = 0
            self.dp_tiles = self.tiles
            self.sk_iters = 0
            self.iters_per_prog = 0
            self.iters_rem = 0

    # -- Stream-K wave -------------------------------------------------------
    def prog_range(self, pid: int):
        """[start, last) of the global iteration index for program ``pid``."""
        q, r = self.iters_per_prog, self.iters_rem
        return pid * q + min(pid, r), (pid + 1) * q + min(pid + 1, r)

    def segments(self, pid: int):
        """(tile, k_begin, k_end) pieces of program ``pid``'s range."""
        start, last = self.prog_range(pid)
        out = []
        while start < last:
            end = min(start + (self.ipt - start % self.ipt), last)
            tile = start // self.ipt
            out.append((tile, start - tile * self.ipt, end - tile * self.ipt))
            start = end
        return out

    def contributors(self):
        """{tile: [(pid, k0, k1), ...] ascending in k} for every Stream-K tile."""
        out: dict[int, list] = {}
        if self.g <= 0:
            return out
        for pid in range(self.g):
            for tile, k0, k1 in self.segments(pid):
                out.setdefault(tile, []).append((pid, k0, k1))
        for tile in out:
            out[tile].sort(key=lambda s: s[1])
        return out

    # -- whole tiles -----------------------------------------------------------
    def whole_tiles(self):
        """Tile ids computed whole, after the Stream-K tiles."""
        return list(range(self.sk_tiles, self.tiles))

    # -- raster ------------------------------------------------------------------
    def coords(self, tile: int):
        """Tile id -> (tile row, tile column)."""
        tm, tn, G = self.tiles_m, self.tiles_n, self.group_m
        if G > 0:
            width = G * tn
            gid = tile // width
            gsize = min(tm - gid * G, G)
            return gid * G + tile % gsize, (tile % width) // gsize
        return tile // tn, tile % tn


def splitk_parts(ipt: int, S: int):
    """k-ranges of a fixed split of one tile's ``ipt`` iterations into ``S``
    parts (the issue's closing comments name split-K as the alternative
    decomposition but print no formula; reading: near-equal contiguous parts,
    part p = [floor(p*ipt/S), floor((p+1)*ipt/S)), the first one the owner)."""
    return [(p * ipt // S, (p + 1) * ipt // S) for p in range(S)]


def cluster_split_units(tiles: int, ipt: int, S: int):
    """Work of each CTA when the S split-K parts of every tile run as one
    thread-block cluster (reading: CTA c takes part c mod S of tile c // S,
    so the CTAs of a cluster -- consecutive indices -- are the parts of one
    tile in ascending k).  Returns [(tile, k_begin, k_end)] indexed by CTA."""
    parts = splitk_parts(ipt, S)
    return [(c // S,) + parts[c % S] for c in range(tiles * S)]


def hilbert_curve(order: int):
    """Cells (x, y) of the Hilbert curve on a 2^order square, in curve order,
    by the recursive construction: the curve of order n is four copies of the
    order n-1 curve -- lower left transposed, upper left, upper right, lower
    right reflected along the anti-diagonal -- joined end to end."""
    if order == 0:
        return [(0, 0)]
    prev = hilbert_curve(order - 1)
    h = 1 << (order - 1)
    q1 = [(y, x) for x, y in prev]                         # transpose
    q2 = [(x, y + h) for x, y in prev]
    q3 = [(x + h, y + h) for x, y in prev]
    q4 = [(2 * h - 1 - y, h - 1 - x) for x, y in prev]     # anti-transpose
    return q1 + q2 + q3 + q4


def hilbert_tiles(tiles_m: int, tiles_n: int):
    """Tile order (row, column) along the Hilbert curve of the smallest
    power-of-two square covering the grid, keeping the cells inside it
    (reading of the blog summary's "Hilbert curves" scheduling policy)."""
    order = 0
    while (1 << order) < max(tiles_m, tiles_n):
        order += 1
    return [(y, x) for x, y in hilbert_curve(order) if y < tiles_m and x < tiles_n]
