"""Pins for the Stream-K schedule oracle: hand-worked examples, closed forms
and exhaustive coverage invariants."""
import os

import pytest

from oracle.streamk_schedule import Schedule, cdiv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "streamk_worked_example.txt")


def _parse_golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        prob, pid, segs = (s.strip() for s in line.split("|"))
        kv = dict(p.split("=") for p in prob.split(","))
        segs = [tuple(int(v) for v in s.split(":")) for s in segs.split()]
        rows.append(({k: int(v) for k, v in kv.items()}, int(pid), segs))
    return rows


def test_hand_worked_examples():
    rows = _parse_golden()
    assert len(rows) == 10
    for prob, pid, segs in rows:
        s = Schedule(prob["M"], prob["N"], prob["K"], 128, 128, 32, prob["g"])
        assert s.segments(pid) == segs, (prob, pid)


@pytest.mark.parametrize(
    "M,N,K,BN,g,tiles,ipt,sk,dp,per,rem",
    [
        # tile counts worked by hand for the five measured workloads, 128 x BN x 64 tiles
        (512, 512, 512, 128, 148, 16, 8, 16, 0, 0, 128),
        (8192, 8192, 8192, 128, 148, 4096, 128, 248, 3848, 214, 72),
        (2304, 2304, 8192, 128, 148, 324, 128, 176, 148, 152, 32),
        (8192, 14336, 4096, 128, 148, 7168, 64, 212, 6956, 91, 100),
        (64, 8192, 8192, 128, 148, 64, 128, 64, 0, 55, 52),
        (8192, 8192, 8192, 256, 152, 2048, 128, 224, 1824, 188, 96),
        (2304, 2304, 8192, 256, 152, 162, 128, 10, 152, 8, 64),
    ],
)
def test_workload_closed_forms(M, N, K, BN, g, tiles, ipt, sk, dp, per, rem):
    s = Schedule(M, N, K, 128, BN, 64, g)
    assert (s.tiles, s.ipt, s.sk_tiles, s.dp_tiles) == (tiles, ipt, sk, dp)
    assert (s.iters_per_prog, s.iters_rem) == (per, rem)
    assert per * g + rem == sk * ipt


def test_two_tiles_off_and_no_streamk():
    s = Schedule(2304, 2304, 8192, 128, 128, 64, 148, two_tiles=False)
    assert s.sk_tiles == 324 % 148 == 28
    s = Schedule(2304, 2304, 8192, 128, 128, 64, 0)
    assert s.sk_tiles == 0 and s.dp_tiles == 324 and s.segments(0) == []


def _check_cover(s: Schedule):
    seen = {}
    for pid in range(s.g):
        segs = s.segments(pid)
        start, last = s.prog_range(pid)
        assert sum(k1 - k0 for _, k0, k1 in segs) == last - start
        # only the first segment may start mid-tile, only the last may end mid-tile
        for idx, (t, k0, k1) in enumerate(segs):
            assert 0 <= k0 < k1 <= s.ipt and 0 <= t < s.sk_tiles
            if idx > 0:
                assert k0 == 0
            if idx < len(segs) - 1:
                assert k1 == s.ipt
            for k in range(k0, k1):
                assert (t, k) not in seen
                seen[(t, k)] = pid
    assert len(seen) == s.sk_tiles * s.ipt
    # contributors of a tile are consecutive programs in ascending k
    for t, parts in s.contributors().items():
        assert parts[0][1] == 0 and parts[-1][2] == s.ipt
        for a, b in zip(parts, parts[1:]):
            assert a[2] == b[1] and b[0] == a[0] + 1
    assert s.whole_tiles() == list(range(s.sk_tiles, s.tiles))
    if s.g > 0:
        assert s.dp_tiles % s.g == 0 or s.dp_tiles < s.g


def test_coverage_exhaustive_small():
    for tiles_m in range(1, 7):
        for tiles_n in range(1, 6):
            for ipt in (1, 2, 3, 5, 8):
                for g in (1, 2, 3, 4, 7, 16, 31):
                    for two in (True, False):
                        s = Schedule(tiles_m * 16, tiles_n * 16, ipt * 8, 16, 16, 8, g, two)
                        _check_cover(s)
                    s = Schedule(tiles_m * 16, tiles_n * 16, ipt * 8, 16, 16, 8, g,
                                 all_streamk=True)
                    assert s.sk_tiles == s.tiles and s.dp_tiles == 0
                    _check_cover(s)


def test_coverage_workloads():
    for (M, N, K, BN) in [(2304, 2304, 8192, 128), (64, 8192, 8192, 128),
                          (512, 512, 512, 128), (2304, 2304, 8192, 256)]:
        for g in (2, 7, 148, 152, 296):
            _check_cover(Schedule(M, N, K, 128, BN, 64, g))


def test_raster_closed_forms():
    for tm in range(1, 20):
        for tn in range(1, 12):
            for G in (0, 1, 2, 3, 8):
                s = Schedule(tm * 128, tn * 128, 64, 128, 128, 64, 0, group_m=G)
                coords = [s.coords(t) for t in range(s.tiles)]
                assert sorted(coords) == [(m, n) for m in range(tm) for n in range(tn)]
                if G in (0, 1):
                    assert coords == [(t // tn, t % tn) for t in range(s.tiles)]
                if G >= tm:
                    assert coords == [(t % tm, t // tm) for t in range(s.tiles)]
    # a hand-worked grouped raster: 3 x 2 tiles, GROUP_M=2
    s = Schedule(384, 256, 64, 128, 128, 64, 0, group_m=2)
    assert [s.coords(t) for t in range(6)] == [(0, 0), (1, 0), (0, 1), (1, 1), (2, 0), (2, 1)]


def test_cdiv():
    assert [cdiv(a, 4) for a in range(0, 10)] == [0, 1, 1, 1, 1, 2, 2, 2, 2, 3]


def test_hilbert_curve_closed_forms():
    from oracle.streamk_schedule import hilbert_curve, hilbert_tiles
    # the order-1 and order-2 curves, written out by hand
    assert hilbert_curve(1) == [(0, 0), (0, 1), (1, 1), (1, 0)]
    assert hilbert_curve(2) == [(0, 0), (1, 0), (1, 1), (0, 1), (0, 2), (0, 3), (1, 3), (1, 2),
                                (2, 2), (2, 3), (3, 3), (3, 2), (3, 1), (2, 1), (2, 0), (3, 0)]
    for order in range(1, 7):
        c = hilbert_curve(order)
        n = 1 << order
        assert sorted(c) == [(x, y) for x in range(n) for y in range(n)]
        # consecutive cells are grid neighbours; the curve runs corner to corner
        assert all(abs(a[0] - b[0]) + abs(a[1] - b[1]) == 1 for a, b in zip(c, c[1:]))
        assert c[0] == (0, 0) and c[-1] == (n - 1, 0)
    t = hilbert_tiles(3, 5)
    assert sorted(t) == [(m, n) for m in range(3) for n in range(5)]


def test_splitk_parts_hand_worked():
    from oracle.streamk_schedule import splitk_parts
    path = os.path.join(os.path.dirname(__file__), "golden", "splitk_parts.txt")
    rows = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, parts = (x.strip() for x in line.split("|"))
        ipt, S = (int(v) for v in head.split())
        want = [tuple(int(v) for v in p.split(":")) for p in parts.split()]
        assert splitk_parts(ipt, S) == want, (ipt, S)
        rows += 1
    assert rows == 7


def test_splitk_parts_cover_the_tile_in_order():
    # contiguous, ascending, non-empty when S <= ipt, sizes differ by at most one
    from oracle.streamk_schedule import splitk_parts
    for ipt in range(1, 70):
        for S in range(1, ipt + 1):
            parts = splitk_parts(ipt, S)
            assert parts[0][0] == 0 and parts[-1][1] == ipt and len(parts) == S
            assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
            sizes = [e - b for b, e in parts]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1


def test_cluster_split_units_hand_worked():
    # two tiles of 10 k-iterations, four parts each (parts from the split-K
    # golden reading: 10/4 = 2.5 -> 2, 20/4 = 5, 30/4 = 7.5 -> 7, 10)
    from oracle.streamk_schedule import cluster_split_units
    assert cluster_split_units(2, 10, 4) == [(0, 0, 2), (0, 2, 5), (0, 5, 7), (0, 7, 10),
                                             (1, 0, 2), (1, 2, 5), (1, 5, 7), (1, 7, 10)]
    # every (tile, k) exactly once, the CTAs of a cluster in ascending k
    for tiles, ipt, S in ((3, 128, 4), (5, 9, 8), (1, 2, 2)):
        units = cluster_split_units(tiles, ipt, S)
        cover = sorted((t, k) for t, k0, k1 in units for k in range(k0, k1))
        assert cover == [(t, k) for t in range(tiles) for k in range(ipt)]
