"""GPU parity of cluster split-K (GEMM_OPT_SPLIT_K_CLUSTER): the S k-parts of
every tile run as one thread-block cluster and add their fp32 partials through
distributed shared memory.

Bar: the acceptance bound against the oracle on every element; bit-exact on
integer-valued inputs; bitwise identical run to run; and bitwise identical to
the workspace form of split-K with the same S, which adds the same partials in
the same ascending-k order."""
import numpy as np
import pytest
import torch

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs
from tests.gpu_util import GUARD, SENTINEL, Workspace, ensure_built, run, to_device

pytestmark = pytest.mark.gpu

LAYOUTS = [(0, 0), (0, 1), (1, 0), (1, 1)]
# (M, N, K, S, tile_n): half-height A (M <= 64) and full tiles, 128- and
# 256-wide, S = 2, 4, 8, ragged M, N and K, parts of unequal length
SHAPES = [(64, 2048, 4096, 4, 256), (64, 1024, 8192, 8, 0), (40, 264, 1000, 2, 128),
          (200, 1000, 2048, 2, 128), (256, 512, 4096, 4, 256), (129, 136, 520, 8, 0),
          (8, 8, 1024, 8, 256), (640, 384, 3000, 4, 128)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    oracle.build()


def _plans(M, N, K, dtype, la, lb, S, tile_n):
    opts = {"split_k": S}
    if tile_n:
        opts["tile_n"] = tile_n
    kc = B.Plan(M, N, K, dtype, la, lb, "splitk", split_cluster=1, **opts)
    # the workspace form on the same tiles (1-CTA MMAs of the same width)
    opts["tile_n"] = kc.info("tile_n")
    ws = B.Plan(M, N, K, dtype, la, lb, "splitk", cluster_m=1, **opts)
    return kc, ws


@pytest.mark.parametrize("dtype", [inputs.F16, inputs.BF16])
@pytest.mark.parametrize("la,lb", LAYOUTS)
@pytest.mark.parametrize("M,N,K,S,tile_n", SHAPES)
def test_cluster_splitk_parity(M, N, K, S, tile_n, dtype, la, lb):
    if la == 1 and M % 8:
        pytest.skip("column-major A needs M a multiple of 8")
    kc, wsp = _plans(M, N, K, dtype, la, lb, S, tile_n)
    assert kc.info("split_k_cluster") == 1 and kc.workspace_size == 0
    assert kc.info("split_k") == S and wsp.info("split_k") == S
    assert kc.info("tile_n") == wsp.info("tile_n")
    ws = Workspace()
    A, Bm = inputs.operands(M, N, K, dtype, la, lb, ("normal", 1.0), ("normal", 1.0), 77)
    dA, dB = to_device(A), to_device(Bm)
    C64, S_abs, _ = oracle.gemm(A, Bm, M, N, K, dtype, la, lb)
    got = run(kc, dA, dB, M, N, ws)
    ok, worst, nbad = oracle.check(got, dtype, C64, S_abs, K)
    assert ok, (nbad, worst)
    assert np.array_equal(run(kc, dA, dB, M, N, ws), got)          # run to run
    assert np.array_equal(run(wsp, dA, dB, M, N, ws), got)         # same sums, same order
    Ai, Bi = inputs.operands(M, N, K, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, 78)
    _, _, Cref = oracle.gemm(Ai, Bi, M, N, K, dtype, la, lb, with_abs=False)
    assert np.array_equal(run(kc, to_device(Ai), to_device(Bi), M, N, ws), Cref)
    kc.close()
    wsp.close()


def test_cluster_splitk_skinny_workload_full_size():
    spec, A, Bm = inputs.workload("skinny64x8192x8192_f16")
    M, N, K, dtype = spec["M"], spec["N"], spec["K"], spec["dtype"]
    p = B.Plan(M, N, K, dtype, 0, 0, "splitk", split_cluster=1)
    assert (p.info("tile_n"), p.info("split_k"), p.info("grid")) == (256, 4, 128)
    C64, S_abs, _ = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0)
    got = run(p, to_device(A), to_device(Bm), M, N)
    ok, worst, nbad = oracle.check(got, dtype, C64, S_abs, K)
    assert ok, (nbad, worst)
    p.close()


def test_cluster_splitk_many_waves_of_clusters():
    # more clusters than fit the GPU at once: they run in waves, independently
    M, N, K, dtype = 2048, 4096, 1024, inputs.BF16
    A, Bm = inputs.operands(M, N, K, dtype, 0, 1, inputs.INT_LAW, inputs.INT_LAW, 79)
    p = B.Plan(M, N, K, dtype, 0, 1, "splitk", split_cluster=1, split_k=4)
    assert p.info("grid") > 4 * p.info("num_sms")
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 1, with_abs=False)
    assert np.array_equal(run(p, to_device(A), to_device(Bm), M, N), Cref)
    p.close()


def test_cluster_splitk_timeout_skips_only_the_waiting_parts():
    # CTA 1 (part 1 of tile 0) signals no one: the other parts of tile 0 give
    # up after the wait limit and store nothing; part 1 itself, which hears
    # from all the others, stores its slice; tile 1 is complete.  The next
    # run is correct.
    M, N, K, dtype, S = 64, 512, 4096, inputs.F16, 4
    A, Bm = inputs.operands(M, N, K, dtype, 0, 0, inputs.INT_LAW, inputs.INT_LAW, 80)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0, with_abs=False)
    dA, dB = to_device(A), to_device(Bm)
    p = B.Plan(M, N, K, dtype, 0, 0, "splitk", split_cluster=1, split_k=S, tile_n=256,
               wait_limit_us=2000, inject_skip_post=1, group_m=0)
    assert p.info("tiles") == 2 and p.units(1)[0][:3] == (0, 16, 32)
    Cbuf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    p.run(dA, dB, Cbuf.data_ptr() + 2 * GUARD)
    assert p.last_status() == B.GEMM_ERR_TIMEOUT
    host = Cbuf.cpu().numpy().view(np.uint16)
    assert (host[:GUARD] == SENTINEL).all() and (host[-GUARD:] == SENTINEL).all()
    C = host[GUARD:GUARD + M * N].reshape(M, N)
    w = 256 // S
    for part in range(S):
        cols = slice(part * w, (part + 1) * w)
        if part == 1:
            assert np.array_equal(C[:, cols], Cref[:, cols])
        else:
            assert (C[:, cols] == SENTINEL).all(), part
    assert np.array_equal(C[:, 256:], Cref[:, 256:])
    p.set_option(B.GEMM_OPT_INJECT_SKIP_POST, -1)
    assert np.array_equal(run(p, dA, dB, M, N), Cref)
    p.close()


@pytest.mark.parametrize("la,lb", [(0, 1), (1, 0)])
def test_cluster_splitk_host_pipeline(la, lb):
    # gemm_run_host over row chunks: every block is a cluster split-K sub-plan
    M, N, K, dtype = 4096, 512, 2048, inputs.BF16
    A, Bm = inputs.operands(M, N, K, dtype, la, lb, inputs.INT_LAW, inputs.INT_LAW, 81)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, la, lb, with_abs=False)
    p = B.Plan(M, N, K, dtype, la, lb, "splitk", split_cluster=1, host_chunks=4)
    assert p.workspace_size == 0 and p.info("host_chunks") == 4
    hA = torch.from_numpy(A.view(np.int16).ravel().copy()).pin_memory()
    hB = torch.from_numpy(Bm.view(np.int16).ravel().copy()).pin_memory()
    dA, dB = torch.empty_like(hA, device="cuda"), torch.empty_like(hB, device="cuda")
    dC = torch.empty(M * N, dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(2):
        hC = torch.full((M * N,), SENTINEL, dtype=torch.int16).pin_memory()
        p.run_host(hA, hB, hC, dA, dB, dC, None, stream)
        assert p.last_status(stream) == B.GEMM_OK
        assert np.array_equal(hC.numpy().view(np.uint16).reshape(M, N), Cref)
    p.close()


# AUTO on a single row of 128-row tiles: cluster split-K when K has more than
# 16 k-blocks and the unsplit tiles fill under 80 % of the SMs, else unsplit
# persistent tiles.  Every element against the oracle, and bit-exact on
# integer-valued inputs, for each branch (fp16, A and B row-major, like the
# skinny workload).
@pytest.mark.parametrize("M,N,K,want_kc", [(64, 4096, 1024, False), (128, 2048, 1000, False),
                                           (16, 1024, 4096, True), (100, 3000, 2112, True),
                                           (64, 16384, 2048, False)])
def test_auto_single_row_parity(M, N, K, want_kc):
    dtype = inputs.F16
    p = B.Plan(M, N, K, dtype, 0, 0, "auto")
    assert p.info("split_k_cluster") == (1 if want_kc else 0), (M, N, K)
    if not want_kc:
        assert p.info("schedule") == B.GEMM_SCHED_PERSISTENT
    ws = Workspace()
    A, Bm = inputs.operands(M, N, K, dtype, 0, 0, ("normal", 1.0), ("normal", 1.0), 91)
    C64, S_abs, _ = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0)
    ok, worst, nbad = oracle.check(run(p, to_device(A), to_device(Bm), M, N, ws), dtype, C64, S_abs, K)
    assert ok, (nbad, worst)
    Ai, Bi = inputs.operands(M, N, K, dtype, 0, 0, inputs.INT_LAW, inputs.INT_LAW, 92)
    _, _, Cref = oracle.gemm(Ai, Bi, M, N, K, dtype, 0, 0, with_abs=False)
    assert np.array_equal(run(p, to_device(Ai), to_device(Bi), M, N, ws), Cref)
    p.close()
