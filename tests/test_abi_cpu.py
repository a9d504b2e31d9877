"""CPU checks of the C-ABI library: it loads, exports every declared entry
point, and its scheduler (the code the kernel runs, enumerated on the host)
matches the oracle's restatement of the Stream-K decomposition unit by unit.
No compute calls: there is no GPU here."""
import ctypes
import os
import re

import pytest

from oracle.streamk_schedule import Schedule
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(gemm_\w+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert sorted(B.SIGNATURES) == names


def test_status_strings(lib):
    for s in range(8):
        assert B.gemm_status_string(s).startswith("GEMM_")
    assert "UNKNOWN" in B.gemm_status_string(99)


def _roles_from_oracle(o: Schedule):
    contrib = o.contributors()
    out = {}
    for pid in range(o.g):
        units = []
        for tile, k0, k1 in o.segments(pid):
            if k0 > 0:
                units.append((tile, k0, k1, B.ROLE_PEER, 0))
            elif k1 == o.ipt:
                units.append((tile, k0, k1, B.ROLE_FULL, 0))
            else:
                units.append((tile, k0, k1, B.ROLE_OWNER, len(contrib[tile]) - 1))
        out[pid] = units
    return out


SHAPES = [
    # the five measured workloads, small ragged cases, degenerate ones
    (512, 512, 512), (8192, 8192, 8192), (2304, 2304, 8192), (8192, 14336, 4096),
    (64, 8192, 8192), (300, 264, 200), (1, 8, 8), (129, 136, 72), (1000, 40, 4096),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("sms", [148, 152])
@pytest.mark.parametrize("tile_n,cm", [(64, 1), (128, 1), (128, 2), (256, 1), (256, 2)])
def test_streamk_units_match_oracle(lib, M, N, K, sms, tile_n, cm):
    for g, two in ((sms, 1), (8, 1), (sms, 0), (2, 1)):
        p = B.Plan(M, N, K, B.GEMM_BF16, 0, 1, "streamk", offline_sms=sms, tile_n=tile_n,
                   grid=g, two_tiles=two, cluster_m=cm)
        gu = g // cm                       # scheduling units: pairs of CTAs when cm == 2
        o = Schedule(M, N, K, 128 * cm, tile_n, 64, gu, two_tiles=bool(two), group_m=8)
        assert p.info("cluster_m") == cm and p.info("tile_m") == 128 * cm
        assert p.info("tiles") == o.tiles and p.info("sk_tiles") == o.sk_tiles
        assert p.info("sk_iters_per_cta") == o.iters_per_prog
        assert p.info("sk_iters_rem") == o.iters_rem
        assert p.info("grid") == gu * cm
        sk_units = _roles_from_oracle(o)
        whole = []
        for c in range(gu * cm):
            got = p.units(c)
            u = c // cm
            n_sk = len(sk_units[u])
            assert got[:n_sk] == sk_units[u], (c, got[:n_sk], sk_units[u])
            rest = [x[0] for x in got[n_sk:]]
            assert all(x[1:] == (0, o.ipt, B.ROLE_FULL, 0) for x in got[n_sk:])
            assert rest == list(range(o.sk_tiles + u, o.tiles, gu))
            if c % cm == 0:
                whole += rest
        assert sorted(whole) == o.whole_tiles()
        ws = p.workspace_size
        if o.sk_tiles:
            # flags for 2g split tiles (the most the hybrid rule makes), then a slot per CTA
            flag_tiles = max(o.sk_tiles, 2 * gu)
            assert ws == -(-flag_tiles * cm * 8 // 256) * 256 + gu * cm * 128 * tile_n * 4
        else:
            assert ws == 0
        p.close()


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("cm", [1, 2])
def test_all_streamk_mode_matches_oracle(lib, M, N, K, cm):
    g = 152
    p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "streamk", offline_sms=g, cluster_m=cm, sk_mode=1)
    o = Schedule(M, N, K, 128 * cm, p.info("tile_n"), 64, g // cm, all_streamk=True)
    assert p.info("sk_tiles") == o.tiles == o.sk_tiles and o.dp_tiles == 0
    sk_units = _roles_from_oracle(o)
    for c in range(p.info("grid")):
        assert p.units(c) == sk_units[c // cm]
    p.close()


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("cm", [1, 2])
def test_splitk_units(lib, M, N, K, cm):
    from oracle.streamk_schedule import splitk_parts
    for S in (0, 1, 2, 3, 5):
        p = B.Plan(M, N, K, B.GEMM_BF16, 0, 1, "splitk", offline_sms=152, cluster_m=cm, split_k=S)
        tiles, ipt, S_got = p.info("tiles"), p.info("iters_per_tile"), p.info("split_k")
        if S:
            assert S_got == min(S, ipt)
        assert 1 <= S_got <= max(1, ipt)
        parts = splitk_parts(ipt, S_got)
        seen = {}
        for c in range(p.info("grid")):
            units = p.units(c)
            roles = [u[3] for u in units]
            # a CTA runs all its peer units before any owner unit
            if B.ROLE_OWNER in roles:
                assert B.ROLE_PEER not in roles[roles.index(B.ROLE_OWNER):]
            for tile, k0, k1, role, npeers in units:
                part = parts.index((k0, k1))
                key = (tile, part)
                if c % cm == 1:
                    assert seen[key] == c - 1      # the pair's second CTA repeats the unit
                    continue
                assert key not in seen
                seen[key] = c
                if S_got == 1:
                    assert role == B.ROLE_FULL
                elif part == 0:
                    assert role == B.ROLE_OWNER and npeers == S_got - 1
                else:
                    assert role == B.ROLE_PEER and npeers == 0
        assert len(seen) == tiles * S_got
        ws = p.workspace_size
        assert (ws == 0) == (S_got == 1)
        p.close()


def test_auto_schedule_choices(lib):
    cases = {  # workload -> (schedule, all tiles in the Stream-K wave)
        (512, 512, 512): (B.GEMM_SCHED_PERSISTENT, 0),
        (8192, 8192, 8192): (B.GEMM_SCHED_STREAMK, 0),
        (2304, 2304, 8192): (B.GEMM_SCHED_STREAMK, 1),
        (8192, 14336, 4096): (B.GEMM_SCHED_STREAMK, 0),
        (64, 8192, 8192): (B.GEMM_SCHED_SPLITK, 0),
        # from the timed sweep of log-sampled shapes
        (3840, 2816, 5888): (B.GEMM_SCHED_STREAMK, 0),
        (768, 6656, 2304): (B.GEMM_SCHED_STREAMK, 1),
        (4352, 512, 5888): (B.GEMM_SCHED_SPLITK, 0),     # cluster split-K fits one wave
        (256, 1792, 6400): (B.GEMM_SCHED_SPLITK, 0),
        (512, 2048, 768): (B.GEMM_SCHED_PERSISTENT, 0),  # fits, but parts of 6 k-blocks
        (512, 5632, 1280): (B.GEMM_SCHED_STREAMK, 1),
        (4608, 5120, 1024): (B.GEMM_SCHED_PERSISTENT, 0),
        # four or more waves: hybrid for long tiles or many waves
        (5120, 5120, 5120): (B.GEMM_SCHED_STREAMK, 0),
        (4096, 8192, 2048): (B.GEMM_SCHED_PERSISTENT, 0),
        (12288, 12288, 2048): (B.GEMM_SCHED_STREAMK, 0),
    }
    for (M, N, K), (sched, mode) in cases.items():
        p = B.Plan(M, N, K, B.GEMM_BF16, 0, 1, "auto", offline_sms=152)
        assert (p.info("schedule"), p.info("sk_mode")) == (sched, mode), (M, N, K)
        assert p.info("split_k_cluster") == (1 if sched == B.GEMM_SCHED_SPLITK else 0), (M, N, K)
        p.close()


def test_auto_single_row_of_tiles(lib):
    # split-K reduced inside clusters when a choice of it fills one wave, K
    # has more than 16 k-blocks and the unsplit 128-wide tiles would fill
    # under 80 % of the SMs
    for M, N, K, bn, S in ((64, 8192, 8192, 256, 4), (16, 1024, 4096, 128, 8),
                           (128, 8192, 16384, 256, 4), (128, 2048, 2048, 128, 8)):
        p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "auto", offline_sms=152)
        assert p.info("schedule") == B.GEMM_SCHED_SPLITK and p.info("split_k_cluster") == 1
        assert (p.info("tile_n"), p.info("split_k"), p.workspace_size) == (bn, S, 0), (M, N, K)
        p.close()
    # unsplit (persistent) tiles when K has 16 k-blocks or fewer, or when the
    # tiles already fill 80 % of the SMs (shapes of the timed single-row sweep
    # where these ran 10-35 % faster than the split)
    for M, N, K in ((128, 8192, 1024), (64, 4096, 1024), (16, 16384, 1024),
                    (128, 16384, 4096), (128, 16384, 16384)):
        p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "auto", offline_sms=152)
        assert (p.info("schedule"), p.info("split_k_cluster")) == (B.GEMM_SCHED_PERSISTENT, 0), (M, N, K)
        p.close()
    # otherwise no cluster split-K: one k-block (nothing to split), a forced
    # pair cluster, or too many tiles for one wave of 2-part clusters
    for M, N, K, opts in ((64, 8192, 64, {}), (64, 8192, 8192, {"cluster_m": 2}),
                          (64, 65536, 4096, {})):
        p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "auto", offline_sms=152, **opts)
        assert p.info("split_k_cluster") == 0 and p.info("schedule") != B.GEMM_SCHED_SPLITK, (M, N, K)
        p.close()
    # the split-K part count of an AUTO plan does not leak into the choice
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "auto", offline_sms=152, split_k=3)
    assert (p.info("split_k_cluster"), p.info("split_k")) == (1, 4)
    p.close()


def test_half_height_a_for_short_m(lib):
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "streamk", offline_sms=148, tile_n=128)
    assert p.info("a_rows_per_stage") == 64 and p.info("stages") == 9
    p.close()
    p = B.Plan(65, 8192, 8192, B.GEMM_F16, 0, 0, "streamk", offline_sms=148, tile_n=128)
    assert p.info("a_rows_per_stage") == 128 and p.info("stages") == 7
    p.close()


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_dp_and_persistent_units(lib, M, N, K):
    o = Schedule(M, N, K, 128, 128, 64, 0)
    p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "dp", offline_sms=148, tile_n=128, cluster_m=1)
    assert p.info("grid") == o.tiles and p.workspace_size == 0
    for c in range(0, o.tiles, max(1, o.tiles // 50)):
        assert p.units(c) == [(c, 0, o.ipt, B.ROLE_FULL, 0)]
    p.close()
    p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "persistent", offline_sms=148, tile_n=128,
               cluster_m=1)
    g = min(148, o.tiles)
    assert p.info("grid") == g and p.workspace_size == 0
    seen = []
    for c in range(g):
        u = p.units(c)
        assert [x[0] for x in u] == list(range(c, o.tiles, g))
        seen += [x[0] for x in u]
    assert sorted(seen) == list(range(o.tiles))
    p.close()


@pytest.mark.parametrize("group_m", [0, 1, 3, 8])
def test_raster_matches_oracle(lib, group_m):
    for M, N in ((2304, 2304), (8192, 14336), (1000, 3000), (64, 8192)):
        o = Schedule(M, N, 64, 128, 128, 64, 0, group_m=group_m)
        p = B.Plan(M, N, 64, B.GEMM_F16, 0, 0, "persistent", offline_sms=148, tile_n=128,
                   group_m=group_m)
        for t in range(o.tiles):
            assert p.tile_coords(t) == o.coords(t)
        p.close()


def test_default_options(lib):
    p = B.Plan(8192, 8192, 8192, B.GEMM_BF16, 0, 1, "streamk", offline_sms=148)
    assert p.info("tile_n") == 256 and p.info("group_m") == 8 and p.info("tile_k") == 64
    assert p.info("cluster_m") == 2 and p.info("tile_m") == 256 and p.info("grid") == 148
    p.close()
    p = B.Plan(8192, 8192, 8192, B.GEMM_BF16, 0, 1, "streamk", offline_sms=148, cluster_m=1)
    assert p.info("tile_m") == 128 and p.info("grid") == 148
    p.close()
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "dp", offline_sms=148)
    assert p.info("tile_n") == 128 and p.info("group_m") == 0 and p.info("tiles") == 64
    assert p.info("a_rows_per_stage") == 64 and p.info("stages") == 9
    assert p.info("l2_prefetch") == 0 and p.info("k_rotate") == 0
    p.close()
    p = B.Plan(512, 512, 512, B.GEMM_F16, 0, 0, "dp", offline_sms=148)
    assert p.info("tile_n") == 64 and p.info("tiles") == 32 and p.info("stages") == 9
    p.close()
    p = B.Plan(2304, 2304, 8192, B.GEMM_BF16, 0, 1, "streamk", offline_sms=152)
    assert p.info("tile_n") == 256 and p.info("cluster_m") == 2 and p.info("tiles") == 81
    p.close()
    with pytest.raises(B.GemmError) as e:
        B.Plan(512, 512, 512, B.GEMM_F16, 0, 0, "dp", offline_sms=148, tile_n=64, cluster_m=2)
    assert e.value.status == B.GEMM_ERR_UNSUPPORTED


def test_argument_errors(lib):
    with pytest.raises(B.GemmError) as e:
        B.gemm_plan_create_offline(-1, 8, 8, 0, 0, 0, 0, 148)
    assert e.value.status == B.GEMM_ERR_INVALID_ARG
    with pytest.raises(B.GemmError) as e:
        B.gemm_plan_create_offline(8, 8, 8, 5, 0, 0, 0, 148)
    assert e.value.status == B.GEMM_ERR_INVALID_ARG
    with pytest.raises(B.GemmError) as e:
        B.gemm_plan_create_offline(8, 8, 8, 0, 0, 0, 0, 0)
    assert e.value.status == B.GEMM_ERR_INVALID_ARG
    p = B.Plan(256, 256, 256, B.GEMM_F16, 0, 0, "streamk", offline_sms=148)
    for key, val, st in ((B.GEMM_OPT_TILE_N, 96, B.GEMM_ERR_UNSUPPORTED),
                         (B.GEMM_OPT_GRID, 149, B.GEMM_ERR_UNSUPPORTED),
                         (B.GEMM_OPT_TWO_TILES, 2, B.GEMM_ERR_UNSUPPORTED),
                         (99, 0, B.GEMM_ERR_INVALID_ARG)):
        with pytest.raises(B.GemmError) as e:
            p.set_option(key, val)
        assert e.value.status == st
    with pytest.raises(B.GemmError) as e:
        p.units(148)
    assert e.value.status == B.GEMM_ERR_INVALID_ARG
    with pytest.raises(B.GemmError) as e:
        p.run(16, 16, 16, 16)
    assert e.value.status == B.GEMM_ERR_NO_DEVICE
    assert B.gemm_last_status(p.handle) == B.GEMM_ERR_NO_DEVICE
    assert lib.gemm_plan_destroy(None) == 0
    p.close()


def test_owner_peer_structure_on_workloads(lib):
    # among a CTA's Stream-K units, only the first may be a PEER and only the last an OWNER
    for M, N, K in SHAPES:
        p = B.Plan(M, N, K, B.GEMM_BF16, 0, 1, "streamk", offline_sms=148)
        sk = p.info("sk_tiles")
        for c in range(p.info("grid")):
            roles = [u[3] for u in p.units(c) if u[0] < sk]
            assert B.ROLE_PEER not in roles[1:]
            assert B.ROLE_OWNER not in roles[:-1]
        p.close()


def test_hilbert_raster_matches_oracle(lib):
    from oracle.streamk_schedule import hilbert_tiles
    for M, N in ((512, 512), (2304, 2304), (8192, 14336), (64, 8192), (1000, 3000), (384, 128)):
        for cm in (1, 2):
            p = B.Plan(M, N, 64, B.GEMM_BF16, 0, 1, "persistent", offline_sms=152, tile_n=128,
                       cluster_m=cm, raster=1)
            assert p.info("raster") == 1
            ref = hilbert_tiles(p.info("tiles_m"), p.info("tiles_n"))
            assert [p.tile_coords(t) for t in range(p.info("tiles"))] == ref
            # units follow the same order
            seen = sorted(u[0] for c in range(0, p.info("grid"), cm) for u in p.units(c))
            assert seen == list(range(p.info("tiles")))
            p.close()


def test_host_chunk_policy(lib):
    """gemm_run_host's block grid: row chunks of whole tile rows and column
    chunks of whole tile columns; quarters of each side when both are long,
    chunks of the long side only otherwise; serial when a side is short and
    no split is asked for, or where the blocks' sub-plans would not fit the
    plan's workspace."""
    def grid(M, N, sched, **opt):
        p = B.Plan(M, N, 4096, B.GEMM_BF16, 0, 1, sched, offline_sms=152, **opt)
        out = (p.info("host_chunks"), p.info("host_col_chunks"), p.info("tile_m"), p.info("tile_n"))
        p.close()
        return out
    # B no larger than A: row chunks, min(8, M / 512)
    assert grid(8192, 8192, "persistent")[:2] == (8, 1)
    assert grid(8192, 8192, "auto")[:2] == (8, 1)
    assert grid(8192, 8192, "streamk")[:2] == (8, 1)       # sub-plans fit the workspace
    assert grid(8192, 8192, "splitk")[:2] == (8, 1)
    assert grid(8192, 1024, "persistent")[:2] == (8, 1)
    # B the larger operand: blocks, min(4, M / 1024) x min(4, N / 1024)
    assert grid(2048, 4096, "persistent")[:2] == (2, 4)
    assert grid(8192, 14336, "streamk")[:2] == (4, 4)
    assert grid(8192, 14336, "auto")[:2] == (4, 4)
    assert grid(64, 8192, "streamk")[:2] == (1, 8)         # only N is long: column chunks
    assert grid(1024, 1024, "persistent")[:2] == (1, 1)    # serial
    assert grid(8192, 8192, "persistent", host_chunks=1)[:2] == (1, 1)
    assert grid(4096, 8192, "persistent", host_chunks=1)[:2] == (1, 4)
    # chunks round up to whole tiles: 1000 rows in 256-row tiles -> 3 chunks of 512 rows become 2
    n, nc, tm, tn = grid(1000, 1000, "persistent", host_chunks=3, host_col_chunks=3, cluster_m=2)
    assert tm == 256 and n == 2 and nc == 3 and tn in (128, 256)
    n, nc, tm, tn = grid(1000, 1024, "persistent", host_chunks=16, host_col_chunks=16, cluster_m=1,
                         tile_n=128)
    assert tm == 128 and tn == 128 and n == 8 and nc == 8
    with pytest.raises(B.GemmError):
        grid(1000, 1000, "persistent", host_chunks=17)
    with pytest.raises(B.GemmError):
        grid(1000, 1000, "persistent", host_col_chunks=17)

@pytest.mark.parametrize("M,N,K", [(64, 8192, 8192), (300, 1000, 2048), (128, 256, 128), (1, 8, 4096)])
def test_cluster_splitk_units_match_oracle(lib, M, N, K):
    from oracle.streamk_schedule import cluster_split_units
    for S in (0, 2, 4, 8):
        try:
            p = B.Plan(M, N, K, B.GEMM_F16, 0, 0, "splitk", offline_sms=152, split_cluster=1,
                       split_k=S)
        except B.GemmError as e:
            assert e.status == B.GEMM_ERR_UNSUPPORTED and S > (K + 63) // 64
            continue
        tiles, ipt, S_got = p.info("tiles"), p.info("iters_per_tile"), p.info("split_k")
        assert p.info("split_k_cluster") == 1 and p.info("cluster_m") == 1
        assert p.info("tile_n") in (128, 256) and p.workspace_size == 0
        if S:
            assert S_got == S
        assert S_got in (2, 4, 8) and S_got <= ipt
        assert p.info("grid") == tiles * S_got
        want = cluster_split_units(tiles, ipt, S_got)
        for c in range(p.info("grid")):
            units = p.units(c)
            assert len(units) == 1
            tile, k0, k1, role, npeers = units[0]
            assert (tile, k0, k1) == want[c]
            assert role == B.ROLE_CLUSTER_PART and npeers == S_got - 1
        p.close()


def test_cluster_splitk_defaults_and_refusals(lib):
    # the skinny workload: 256-wide tiles, the most parts that keep one wave
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "splitk", offline_sms=152, split_cluster=1)
    assert (p.info("tile_n"), p.info("split_k"), p.info("grid")) == (256, 4, 128)
    assert p.info("a_rows_per_stage") == 64 and p.info("schedule") == B.GEMM_SCHED_SPLITK
    p.close()
    # few tiles: 128-wide tiles when they put more CTAs in the wave (8 x 8
    # against 4 x 8 at 256 wide)
    p = B.Plan(128, 1024, 4096, B.GEMM_F16, 0, 0, "splitk", offline_sms=152, split_cluster=1)
    assert (p.info("tile_n"), p.info("split_k"), p.info("grid")) == (128, 8, 64)
    p.close()
    # a tie (20 tiles x 4 parts or 40 x 2) goes to 256-wide tiles
    p = B.Plan(64, 5120, 4096, B.GEMM_F16, 0, 0, "splitk", offline_sms=152, split_cluster=1)
    assert (p.info("tile_n"), p.info("split_k"), p.info("grid")) == (256, 4, 80)
    p.close()
    # a wide product: no pair fits one wave, so 256-wide tiles and 2 parts
    p = B.Plan(256, 20480, 4096, B.GEMM_BF16, 0, 1, "splitk", offline_sms=152, split_cluster=1)
    assert (p.info("tile_n"), p.info("split_k"), p.info("grid")) == (256, 2, 320)
    p.close()
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "splitk", offline_sms=152)
    for key, val in ((B.GEMM_OPT_SPLIT_K, 3), (B.GEMM_OPT_TILE_N, 64), (B.GEMM_OPT_CLUSTER_M, 2)):
        q = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "splitk", offline_sms=152)
        q.set_option(key, val)
        with pytest.raises(B.GemmError) as e:
            q.set_option(B.GEMM_OPT_SPLIT_K_CLUSTER, 1)
        assert e.value.status == B.GEMM_ERR_UNSUPPORTED
        assert q.info("split_k_cluster") == 0          # the plan keeps its options
        q.close()
    with pytest.raises(B.GemmError):
        p.set_option(B.GEMM_OPT_SPLIT_K_CLUSTER, 2)
    p.close()
    # other schedules ignore the option
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "streamk", offline_sms=152, split_cluster=1)
    assert p.info("split_k_cluster") == 0 and p.workspace_size > 0
    p.close()


def test_early_prefetch_default_and_option(lib):
    # 8 k-blocks when the launch fills at least 3/4 of the SMs, else none
    for shape, want in (((64, 8192, 8192), 8), ((16, 1024, 4096), 0), ((8192, 8192, 8192), 8),
                        ((2304, 2304, 8192), 8), ((512, 512, 512), 0)):
        p = B.Plan(*shape, B.GEMM_F16, 0, 0, "auto", offline_sms=152)
        ctas = p.info("grid")
        assert p.info("early_prefetch") == want == (8 if 4 * ctas >= 3 * 152 else 0), shape
        p.close()
    p = B.Plan(64, 8192, 8192, B.GEMM_F16, 0, 0, "auto", offline_sms=152, early_prefetch=3)
    assert p.info("early_prefetch") == 3
    p.set_option(B.GEMM_OPT_EARLY_PREFETCH, 0)
    assert p.info("early_prefetch") == 0
    p.set_option(B.GEMM_OPT_EARLY_PREFETCH, -1)
    assert p.info("early_prefetch") == 8
    for bad in (-2, 257):
        with pytest.raises(B.GemmError) as e:
            p.set_option(B.GEMM_OPT_EARLY_PREFETCH, bad)
        assert e.value.status == B.GEMM_ERR_UNSUPPORTED
    p.close()
