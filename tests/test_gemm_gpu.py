"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bar: every element within |C - C_ref| <= 2^-8 |C_ref| + K 2^-22 sum|a||b|;
bit-exact on integer-valued inputs; bitwise identical from run to run."""
import numpy as np
import pytest
import torch

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs
from tests.gpu_util import Workspace, ensure_built, run, to_device

pytestmark = pytest.mark.gpu

SCHEDS = ["dp", "persistent", "streamk", "splitk", "auto"]
# (tile width, CTAs per cluster, pair MMA): every kernel variant
CONFIGS = [(64, 1, 0), (128, 1, 0), (128, 2, 0), (128, 2, 1), (256, 1, 0), (256, 2, 0),
           (256, 2, 1)]
LAYOUTS = [(0, 0), (0, 1), (1, 0), (1, 1)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    oracle.build()


def _case(M, N, K, dtype, la, lb, law, seed):
    A, Bm = inputs.operands(M, N, K, dtype, la, lb, law, law, seed)
    return A, Bm, to_device(A), to_device(Bm)


def _check_full(Cb, A, Bm, M, N, K, dtype, la, lb, exact=False):
    C64, S, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
    if exact:
        assert np.array_equal(Cb, Cref), "integer inputs must be bit-exact"
    ok, worst, nbad = oracle.check(Cb, dtype, C64, S, K)
    assert ok, "%d elements outside the bound (worst ratio %.3g)" % (nbad, worst)
    return Cref


# ------------------------------------------------------------------ small shapes
SMALL = [(300, 264, 200), (129, 136, 72), (257, 520, 1000), (1, 8, 8), (64, 512, 4096),
         (128, 256, 64), (640, 384, 520)]


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
@pytest.mark.parametrize("la,lb", LAYOUTS)
def test_parity_small(sched, dtype, la, lb):
    ws = Workspace()
    for i, (M, N, K) in enumerate(SMALL):
        if la == 1 and M % 8:
            continue
        A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, ("normal", 1.0), 10 + i)
        for tile_n, cm, pair in CONFIGS:
            p = B.Plan(M, N, K, dtype, la, lb, sched, tile_n=tile_n, cluster_m=cm,
                       pair_mma=pair)
            Cb = run(p, dA, dB, M, N, ws)
            _check_full(Cb, A, Bm, M, N, K, dtype, la, lb)
            p.close()


@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
@pytest.mark.parametrize("la,lb", LAYOUTS)
def test_integer_bit_exact_small(sched, dtype, la, lb):
    ws = Workspace()
    for i, (M, N, K) in enumerate(SMALL):
        if la == 1 and M % 8:
            continue
        A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, inputs.INT_LAW, 50 + i)
        for cm, pair in ((1, 0), (2, 0), (2, 1)):
            p = B.Plan(M, N, K, dtype, la, lb, sched, cluster_m=cm, pair_mma=pair)
            Cb = run(p, dA, dB, M, N, ws)
            _check_full(Cb, A, Bm, M, N, K, dtype, la, lb, exact=True)
            p.close()


@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
def test_streamk_forced_grids_integer(dtype):
    # several contributors per tile; every grid must give the oracle's bits
    M, N, K = 384, 512, 2048
    A, Bm, dA, dB = _case(M, N, K, dtype, 0, 0, inputs.INT_LAW, 7)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ws = Workspace()
    for tile_n, cm, pair in CONFIGS:
        tiles = -(-3 // cm) * (N // tile_n)
        for g in sorted({2, 8, 14, tiles * cm, sms}):
            for two in (0, 1):
                p = B.Plan(M, N, K, dtype, 0, 0, "streamk", tile_n=tile_n, grid=g,
                           two_tiles=two, cluster_m=cm, pair_mma=pair)
                Cb = run(p, dA, dB, M, N, ws)
                assert np.array_equal(Cb, Cref), (tile_n, cm, pair, g, two)
                p.close()


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("sched", SCHEDS)
def test_pair_mma(tile_n, sched):
    # 2-CTA clusters issuing one tcgen05 pair MMA (256 x BN) per k-step
    ws = Workspace()
    for i, (M, N, K) in enumerate(((256, 256, 512), (300, 264, 200), (512, 640, 1032),
                                   (1000, 1040, 2048), (64, 1024, 2048), (40, 512, 1032))):
        for dtype in (inputs.F16, inputs.BF16):
            for la, lb in LAYOUTS:
                if la == 1 and M % 8:
                    continue
                for law in (inputs.INT_LAW, ("normal", 1.0)):
                    A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, law, 60 + i)
                    p = B.Plan(M, N, K, dtype, la, lb, sched, tile_n=tile_n, cluster_m=2,
                               pair_mma=1)
                    assert p.info("pair_mma") == 1 and p.info("tile_m") == 256
                    assert p.info("a_rows_per_stage") == (64 if M <= 64 else 128)
                    Cb = run(p, dA, dB, M, N, ws)
                    _check_full(Cb, A, Bm, M, N, K, dtype, la, lb,
                                exact=law == inputs.INT_LAW)
                    assert np.array_equal(run(p, dA, dB, M, N, ws), Cb)
                    p.close()


@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
def test_all_streamk_mode_and_short_m(dtype):
    ws = Workspace()
    for (M, N, K), la, lb in (((384, 1024, 2048), 0, 1), ((64, 2048, 3000 // 8 * 8), 0, 0),
                              ((40, 520, 1032), 0, 1), ((64, 1024, 1024), 1, 0)):
        A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, inputs.INT_LAW, 15)
        _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
        for cm in (1, 2):
            for mode in (0, 1):
                p = B.Plan(M, N, K, dtype, la, lb, "streamk", cluster_m=cm, sk_mode=mode)
                if M <= 64 and cm == 1 and p.info("tile_n") == 128:
                    assert p.info("a_rows_per_stage") == 64
                first = run(p, dA, dB, M, N, ws)
                assert np.array_equal(first, Cref), (M, N, K, cm, mode)
                assert np.array_equal(run(p, dA, dB, M, N, ws), first)
                p.close()


@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
def test_owner_stages_all_peers_when_c_does_not_fit_beside_them(dtype):
    # 64 rows, 256-wide tiles, four contributors per tile: the owner's three
    # peer partials fill the 200 KB ring, so C is stored straight from registers
    M, N, K = 64, 1024, 2048
    ws = Workspace()
    for la, lb in ((0, 0), (0, 1)):
        A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, inputs.INT_LAW, 48)
        _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
        for g in (16, 12, 20):
            p = B.Plan(M, N, K, dtype, la, lb, "streamk", tile_n=256, cluster_m=1, grid=g)
            assert p.info("a_rows_per_stage") == 64 and p.info("tiles") == 4
            npeers = max(u[4] for c in range(g) for u in p.units(c))
            assert npeers >= 3 or g != 16
            got = run(p, dA, dB, M, N, ws)
            assert np.array_equal(got, Cref), (la, lb, g)
            assert np.array_equal(run(p, dA, dB, M, N, ws), got)
            p.close()


@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
def test_splitk_parts_integer_exact(dtype):
    ws = Workspace()
    for (M, N, K), la, lb in (((384, 1024, 2048), 0, 1), ((64, 2048, 3000 // 8 * 8), 0, 0),
                              ((300, 264, 1000), 1 if 300 % 8 == 0 else 0, 0)):
        A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, inputs.INT_LAW, 16)
        _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
        for cm in (1, 2):
            for S in (0, 2, 3, 7):
                p = B.Plan(M, N, K, dtype, la, lb, "splitk", cluster_m=cm, split_k=S)
                first = run(p, dA, dB, M, N, ws)
                assert np.array_equal(first, Cref), (M, N, K, cm, S)
                assert np.array_equal(run(p, dA, dB, M, N, ws), first)
                p.close()


@pytest.mark.parametrize("sched", SCHEDS)
def test_k_rotation_and_l2_prefetch(sched):
    # whole tiles visiting their k-blocks in rotated order, and B prefetched
    # into L2 ahead of the ring: same bits on integers, within the bound on
    # real values, deterministic
    ws = Workspace()
    for (M, N, K, dtype, la, lb) in ((64, 1024, 2048, inputs.F16, 0, 0),
                                     (300, 520, 1000, inputs.BF16, 0, 1),
                                     (256, 512, 4096, inputs.BF16, 1, 1)):
        for law in (inputs.INT_LAW, ("normal", 1.0)):
            A, Bm, dA, dB = _case(M, N, K, dtype, la, lb, law, 17)
            for tile_n, cm, rot, pf in ((64, 1, 1, 0), (128, 1, 1, 8), (128, 2, 0, 16),
                                        (256, 2, 1, 4)):
                p = B.Plan(M, N, K, dtype, la, lb, sched, tile_n=tile_n, cluster_m=cm,
                           k_rotate=rot, l2_prefetch=pf)
                assert p.info("k_rotate") == rot and p.info("l2_prefetch") == pf
                Cb = run(p, dA, dB, M, N, ws)
                _check_full(Cb, A, Bm, M, N, K, dtype, la, lb, exact=law == inputs.INT_LAW)
                assert np.array_equal(run(p, dA, dB, M, N, ws), Cb)
                p.close()


@pytest.mark.parametrize("sched", SCHEDS)
def test_hilbert_raster(sched):
    ws = Workspace()
    for (M, N, K), cm in (((1000, 1040, 1032), 1), ((768, 1536, 2048), 2), ((64, 1024, 1024), 1)):
        A, Bm, dA, dB = _case(M, N, K, inputs.BF16, 0, 1, inputs.INT_LAW, 18)
        _, _, Cref = oracle.gemm(A, Bm, M, N, K, inputs.BF16, 0, 1)
        p = B.Plan(M, N, K, inputs.BF16, 0, 1, sched, cluster_m=cm, raster=1)
        assert p.info("raster") == 1
        assert np.array_equal(run(p, dA, dB, M, N, ws), Cref)
        p.close()


def test_streamk_deterministic_and_within_bound():
    M, N, K, dtype = 512, 768, 3000 // 8 * 8, inputs.BF16
    A, Bm, dA, dB = _case(M, N, K, dtype, 0, 1, ("normal", 1.0), 8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ws = Workspace()
    for g in (5, sms):
        p = B.Plan(M, N, K, dtype, 0, 1, "streamk", tile_n=128, grid=g)
        first = run(p, dA, dB, M, N, ws)
        _check_full(first, A, Bm, M, N, K, dtype, 0, 1)
        for _ in range(10):
            assert np.array_equal(run(p, dA, dB, M, N, ws), first)
        p.close()


def test_schedules_agree_on_integers():
    M, N, K, dtype = 520, 1000, 1032, inputs.F16
    A, Bm, dA, dB = _case(M, N, K, dtype, 0, 0, inputs.INT_LAW, 9)
    outs = []
    for s in SCHEDS:
        for cm in (1, 2):
            p = B.Plan(M, N, K, dtype, 0, 0, s, cluster_m=cm)
            outs.append(run(p, dA, dB, M, N))
            p.close()
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


# ------------------------------------------------------------------ edge cases
def test_k_zero_gives_zero_and_empty_is_noop():
    p = B.Plan(100, 64, 0, inputs.F16, 0, 0, "streamk")
    dA = torch.zeros(8, dtype=torch.int16, device="cuda")
    Cb = run(p, dA, dA, 100, 64)
    assert not Cb.any()
    p.close()
    for M, N in ((0, 64), (64, 0)):
        p = B.Plan(M, N, 64, inputs.F16, 0, 0, "streamk")
        p.run(0, 0, 0, None)
        assert p.last_status() == B.GEMM_OK
        p.close()


def test_unsupported_alignment_and_strides():
    p = B.Plan(64, 64, 64, inputs.F16, 0, 0, "dp")
    buf = torch.zeros(64 * 64 + 8, dtype=torch.int16, device="cuda")
    with pytest.raises(B.GemmError) as e:
        p.run(buf.data_ptr() + 2, buf, buf)
    assert e.value.status == B.GEMM_ERR_UNSUPPORTED
    p.close()
    p = B.Plan(64, 64, 60, inputs.F16, 0, 0, "dp")
    with pytest.raises(B.GemmError) as e:
        p.run(buf, buf, buf)
    assert e.value.status == B.GEMM_ERR_UNSUPPORTED
    p.close()
    p = B.Plan(64, 512, 512, inputs.F16, 0, 0, "streamk")
    assert p.workspace_size > 0
    with pytest.raises(B.GemmError) as e:
        p.run(buf, buf, buf, None)
    assert e.value.status == B.GEMM_ERR_WORKSPACE
    p.close()


def test_timeout_is_reported_and_gpu_stays_healthy():
    # a peer that never posts: its owner's bounded wait must run out, the
    # tile's C must stay untouched, and the next run must be correct
    M, N, K, dtype = 128, 128, 4096, inputs.F16
    A, Bm, dA, dB = _case(M, N, K, dtype, 0, 0, inputs.INT_LAW, 11)
    p = B.Plan(M, N, K, dtype, 0, 0, "streamk", tile_n=128, grid=4, wait_limit_us=2000)
    units = [p.units(c) for c in range(4)]
    assert units[0][0][3] == B.ROLE_OWNER and units[1][0][3] == B.ROLE_PEER
    p.set_option(B.GEMM_OPT_INJECT_SKIP_POST, 1)
    ws = Workspace()
    with pytest.raises(B.GemmError) as e:
        run(p, dA, dB, M, N, ws)
    assert e.value.status == B.GEMM_ERR_TIMEOUT
    # C untouched: run again by hand and look at the sentinel
    from tests.gpu_util import GUARD, SENTINEL
    Cbuf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    p.run(dA, dB, Cbuf.data_ptr() + 2 * GUARD, ws.get(p.workspace_size))
    assert p.last_status() == B.GEMM_ERR_TIMEOUT
    assert (Cbuf.cpu().numpy().view(np.uint16) == SENTINEL).all()
    assert p.last_status() == B.GEMM_OK  # cleared by the previous read
    p.set_option(B.GEMM_OPT_INJECT_SKIP_POST, -1)
    Cb = run(p, dA, dB, M, N, ws)
    _check_full(Cb, A, Bm, M, N, K, dtype, 0, 0, exact=True)
    p.close()


def test_timeout_with_clusters_hits_only_the_silent_half():
    # pairs of CTAs: the peer CTA 2 (unit 1, lower half) stays silent, so only
    # the lower half's owner (CTA 0) gives up; the upper half completes
    M, N, K, dtype = 256, 128, 4096, inputs.F16
    A, Bm, dA, dB = _case(M, N, K, dtype, 0, 0, inputs.INT_LAW, 13)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0)
    p = B.Plan(M, N, K, dtype, 0, 0, "streamk", tile_n=128, grid=8, cluster_m=2,
               wait_limit_us=2000, inject_skip_post=2)
    assert p.info("tile_m") == 256 and p.info("grid") == 8
    assert p.units(0)[0][3] == B.ROLE_OWNER and p.units(2)[0][3] == B.ROLE_PEER
    from tests.gpu_util import GUARD, SENTINEL
    ws = Workspace()
    Cbuf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    p.run(dA, dB, Cbuf.data_ptr() + 2 * GUARD, ws.get(p.workspace_size))
    assert p.last_status() == B.GEMM_ERR_TIMEOUT
    host = Cbuf.cpu().numpy().view(np.uint16)[GUARD:GUARD + M * N].reshape(M, N)
    assert (host[:128] == SENTINEL).all()
    assert np.array_equal(host[128:], Cref[128:])
    p.set_option(B.GEMM_OPT_INJECT_SKIP_POST, -1)
    assert np.array_equal(run(p, dA, dB, M, N, ws), Cref)
    p.close()


@pytest.mark.parametrize("sched", SCHEDS)
def test_trace_stamps_are_ordered(sched):
    M, N, K, dtype = 1024, 1536, 1024, inputs.BF16
    A, Bm, dA, dB = _case(M, N, K, dtype, 0, 1, ("normal", 1.0), 14)
    p = B.Plan(M, N, K, dtype, 0, 1, sched)
    ctas = p.info("grid")
    buf = torch.zeros(B.TRACE_STAMPS * ctas, dtype=torch.int64, device="cuda")
    p.set_trace(buf, buf.numel() * 8)
    Cb = run(p, dA, dB, M, N)
    _check_full(Cb, A, Bm, M, N, K, dtype, 0, 1)
    t = buf.cpu().numpy().reshape(ctas, B.TRACE_STAMPS)
    assert (t > 0).all()
    assert (t[:, 0] <= t[:, 1]).all() and (t[:, 1] <= t[:, 2]).all() and (t[:, 2] <= t[:, 3]).all()
    assert t[:, 3].max() - t[:, 0].min() < 10_000_000_000   # one run, well under 10 s
    # the SM cycle counter moves forward over every CTA's lifetime
    assert (t[:, 5] > t[:, 4]).all()
    p.set_trace(None, 0)
    p.close()


@pytest.mark.parametrize("la,lb", [(0, 1), (1, 0)])
def test_run_host_pipelined_chunks(la, lb):
    # row chunks of A in, chunks of C computed and copied out while the next
    # chunk's copy runs; a ragged last chunk; the same bytes as gemm_run
    M, N, K, dtype = 1000, 520, 776, inputs.BF16
    A, Bm = inputs.operands(M, N, K, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, 46)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
    hA = torch.from_numpy(A.view(np.int16).ravel()).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16).ravel()).pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()
    for sched, chunks, opts in (("persistent", 3, {}), ("dp", 4, {}), ("persistent", 16, {}),
                                ("persistent", 1, {}), ("streamk", 3, {}),
                                ("streamk", 4, {"sk_mode": 1}), ("splitk", 3, {})):
        p = B.Plan(M, N, K, dtype, la, lb, sched, host_chunks=chunks, **opts)
        tm = p.info("tile_m")
        rows = -(-(-(-M // chunks)) // tm) * tm          # whole tiles per chunk
        want = 1 if chunks == 1 else -(-M // rows)
        assert p.info("host_chunks") in (want, 1), (sched, chunks)
        if sched in ("persistent", "dp"):
            assert p.info("host_chunks") == want
        for _ in range(2):   # the second call reuses the pipeline
            hC = torch.full((M * N,), 0x7E5A, dtype=torch.int16).pin_memory()
            p.run_host(hA, hB, hC, dA, dB, dC, None if not p.workspace_size else
                       torch.zeros(p.workspace_size, dtype=torch.uint8, device="cuda"), stream)
            assert p.last_status(stream) == B.GEMM_OK
            assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref), (sched, chunks)
        p.close()


@pytest.mark.parametrize("la,lb", LAYOUTS)
def test_run_host_block_grid(la, lb):
    # an nr x nc grid of blocks: column chunks of B (strided copies and a
    # strided tensor map for a row-major B), blocks of C written with the full
    # row stride and copied out as strided rectangles; ragged last blocks
    M, N, K, dtype = 1000, 1040, 776, inputs.F16
    A, Bm = inputs.operands(M, N, K, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, 51)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
    hA = torch.from_numpy(A.view(np.int16).ravel()).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16).ravel()).pin_memory()
    dA, dB = hA.cuda(), hB.cuda()
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()
    for sched, opts in (("persistent", {}), ("streamk", {}), ("streamk", {"sk_mode": 1}),
                        ("splitk", {}), ("dp", {"cluster_m": 1, "tile_n": 128})):
        p = B.Plan(M, N, K, dtype, la, lb, sched, host_chunks=3, host_col_chunks=3, **opts)
        assert p.info("host_chunks") * p.info("host_col_chunks") > 1, (sched, opts)
        w = torch.zeros(max(1, p.workspace_size), dtype=torch.uint8, device="cuda")
        for _ in range(2):
            hC = torch.full((M * N,), 0x7E5A, dtype=torch.int16).pin_memory()
            p.run_host(hA, hB, hC, dA, dB, dC, w if p.workspace_size else None, stream)
            assert p.last_status(stream) == B.GEMM_OK
            assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref), (sched, opts)
        # the device copy of C is left in its row-major layout
        assert np.array_equal(dC.cpu().numpy().view(np.uint16).reshape(M, N), Cref)
        p.close()
    # the automatic grid when B is the larger operand: 2 x 4 blocks
    M, N = 2048, 4096
    A, Bm = inputs.operands(M, N, 256, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, 52)
    _, _, Cref = oracle.gemm(A, Bm, M, N, 256, dtype, la, lb)
    p = B.Plan(M, N, 256, dtype, la, lb, "auto")
    assert (p.info("host_chunks"), p.info("host_col_chunks")) == (2, 4)
    hA = torch.from_numpy(A.view(np.int16).ravel()).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16).ravel()).pin_memory()
    hC = torch.empty(M * N, dtype=torch.int16).pin_memory()
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    w = torch.zeros(max(1, p.workspace_size), dtype=torch.uint8, device="cuda")
    p.run_host(hA, hB, hC, hA.cuda(), hB.cuda(), dC, w if p.workspace_size else None, stream)
    assert p.last_status(stream) == B.GEMM_OK
    assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref)
    p.close()


def test_run_host_splitk_chunks_keep_the_parents_part_count():
    # a split-K plan with one part per tile needs no workspace; its row-chunk
    # sub-plans keep that part count (found by a randomized parity sweep: they
    # used to pick more parts and ask for a workspace the caller never sized)
    M, N, K, dtype = 1000, 592, 2368, inputs.BF16
    A, Bm = inputs.operands(M, N, K, dtype, 0, 0, inputs.INT_LAW, inputs.INT_LAW, 49)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0)
    hA = torch.from_numpy(A.view(np.int16).ravel()).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16).ravel()).pin_memory()
    dA, dB = hA.cuda(), hB.cuda()
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()
    p = B.Plan(M, N, K, dtype, 0, 0, "splitk", group_m=1, host_chunks=2)
    assert p.info("split_k") == 1 and p.workspace_size == 0 and p.info("host_chunks") == 2
    hC = torch.full((M * N,), 0x7E5A, dtype=torch.int16).pin_memory()
    p.run_host(hA, hB, hC, dA, dB, dC, None, stream)
    assert p.last_status(stream) == B.GEMM_OK
    assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref)
    p.close()


def test_run_host_pipeline_follows_options_and_shares_the_workspace():
    # a Stream-K plan: pipelined host runs, device runs and an option change in
    # between, all on one workspace; every result exact
    M, N, K, dtype = 2048, 768, 1024, inputs.F16
    A, Bm = inputs.operands(M, N, K, dtype, 0, 0, inputs.INT_LAW, inputs.INT_LAW, 47)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0)
    hA = torch.from_numpy(A.view(np.int16).ravel()).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16).ravel()).pin_memory()
    dA, dB = hA.cuda(), hB.cuda()
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()
    p = B.Plan(M, N, K, dtype, 0, 0, "streamk", sk_mode=1)
    assert p.info("host_chunks") == 4 and p.workspace_size > 0
    w = torch.zeros(p.workspace_size, dtype=torch.uint8, device="cuda")
    for step in range(6):
        if step == 3:
            p.set_option(B.GEMM_OPT_HOST_CHUNKS, 3)   # the pipeline is rebuilt
            assert p.info("host_chunks") in (2, 3)
        hC = torch.full((M * N,), 0x7E5A, dtype=torch.int16).pin_memory()
        p.run_host(hA, hB, hC, dA, dB, dC, w, stream)
        assert p.last_status(stream) == B.GEMM_OK
        assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref), step
        dC.fill_(0x7E5A)
        p.run(dA, dB, dC, w, stream)
        assert p.last_status(stream) == B.GEMM_OK
        assert np.array_equal(dC.cpu().numpy().view(np.uint16).reshape(M, N), Cref), step
    p.close()


def test_run_host_end_to_end():
    M, N, K, dtype = 256, 384, 640, inputs.BF16
    A, Bm = inputs.operands(M, N, K, dtype, 0, 1, ("normal", 1.0), ("normal", 1.0), 12)
    hA = torch.from_numpy(A.view(np.int16)).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16)).pin_memory()
    hC = torch.empty(M * N, dtype=torch.int16).pin_memory()
    dA = torch.empty_like(hA, device="cuda")
    dB = torch.empty_like(hB, device="cuda")
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    p = B.Plan(M, N, K, dtype, 0, 1, "streamk")
    ws = Workspace()
    stream = torch.cuda.current_stream()
    p.run_host(hA, hB, hC, dA, dB, dC, ws.get(p.workspace_size), stream)
    assert p.last_status(stream) == B.GEMM_OK
    Cb = hC.numpy().view(np.uint16).reshape(M, N)
    _check_full(Cb, A, Bm, M, N, K, dtype, 0, 1)
    p.close()


@pytest.mark.parametrize("sched", ["streamk", "splitk", "persistent"])
def test_chained_products_read_the_previous_output(sched):
    # C1 = A1 B1, then at once C2 = A2 C1 in the same stream: the second launch
    # starts while the first drains (programmatic dependent launch) and
    # prefetches its operands into L2 before waiting for it, yet it must read
    # the C1 that the first product wrote.  Integer inputs keep C2 exact: C1
    # holds integers, and every partial sum of C2 stays below 2^24.
    M1, N1, K1, dt = 512, 1024, 2048, inputs.BF16
    M2 = 384
    ws = Workspace()
    p1 = B.Plan(M1, N1, K1, dt, 0, 1, "streamk")
    p2 = B.Plan(M2, N1, M1, dt, 0, 0, sched, early_prefetch=8)
    stream = torch.cuda.current_stream()
    for rep in range(3):
        A1, B1 = inputs.operands(M1, N1, K1, dt, 0, 1, inputs.INT_LAW, inputs.INT_LAW, 90 + rep)
        A2 = inputs.matrix(M2, M1, 0, dt, inputs.INT_LAW, 95 + rep, 1)
        dA1, dB1, dA2 = to_device(A1), to_device(B1), to_device(A2)
        C1 = torch.empty(M1 * N1, dtype=torch.int16, device="cuda")
        C2 = torch.empty(M2 * N1, dtype=torch.int16, device="cuda")
        w1 = ws.get(p1.workspace_size)
        w2 = torch.zeros(max(1, p2.workspace_size), dtype=torch.uint8, device="cuda")
        p1.run(dA1, dB1, C1, w1, stream)
        p2.run(dA2, C1, C2, w2 if p2.workspace_size else None, stream)
        assert p2.last_status(stream) == B.GEMM_OK and p1.last_status(stream) == B.GEMM_OK
        c1 = C1.cpu().numpy().view(np.uint16).reshape(M1, N1)
        _, _, ref1 = oracle.gemm(A1, B1, M1, N1, K1, dt, 0, 1, with_abs=False)
        assert np.array_equal(c1, ref1)
        _, _, ref2 = oracle.gemm(A2, c1, M2, N1, M1, dt, 0, 0, with_abs=False)
        assert np.array_equal(C2.cpu().numpy().view(np.uint16).reshape(M2, N1), ref2), rep
    p1.close()
    p2.close()


@pytest.mark.parametrize("sched,opts", [("streamk", {}), ("streamk", {"sk_mode": 1}), ("dp", {}),
                                        ("splitk", {"split_cluster": 1})])
def test_early_prefetch_changes_no_bit(sched, opts):
    M, N, K, dt = 1024, 1536, 4096, inputs.BF16
    A, Bm, dA, dB = _case(M, N, K, dt, 0, 1, ("normal", 1.0), 23)
    ws = Workspace()
    outs = []
    for d in (0, 8, 64):
        p = B.Plan(M, N, K, dt, 0, 1, sched, early_prefetch=d, **opts)
        outs.append(run(p, dA, dB, M, N, ws))
        p.close()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    _check_full(outs[0], A, Bm, M, N, K, dt, 0, 1)
