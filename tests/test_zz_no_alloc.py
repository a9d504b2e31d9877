"""gemm_run_no_alloc: the entry point for callers that cannot allocate device
memory (for example a plug-in inside a framework that owns every byte of
device memory and forbids allocation while it runs).  It keeps the Stream-K
and split-K scratch (flags and partial tiles) in the library's fixed device
array instead of a caller workspace.

It runs the same kernel as gemm_run, and the kernel is deterministic, so its
output must equal gemm_run's bit for bit, on consecutive calls and when plans
with different flag layouts take turns in the shared array.  This file is
collected last, and each test builds everything it needs, so it passes both
alone in a fresh process and after the rest of the suite."""
import numpy as np
import pytest
import torch

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs
from tests.gpu_util import GUARD, SENTINEL, ensure_built, run, to_device

pytestmark = pytest.mark.gpu


def _no_alloc(plan, dA, dB, M, N):
    """C through gemm_run_no_alloc, with guard bands around C."""
    Cbuf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    B.gemm_run_no_alloc(plan.handle, dA, dB, Cbuf.data_ptr() + 2 * GUARD)
    assert plan.last_status() == B.GEMM_OK
    host = Cbuf.cpu().numpy().view(np.uint16)
    assert (host[:GUARD] == SENTINEL).all() and (host[-GUARD:] == SENTINEL).all()
    return host[GUARD:GUARD + M * N].reshape(M, N).copy()


def _case(M, N, K, dtype, la, lb, law, seed, sched, **opts):
    A, Bm = inputs.operands(M, N, K, dtype, la, lb, law, law, seed)
    p = B.Plan(M, N, K, dtype, la, lb, sched, **opts)
    assert 0 < p.workspace_size <= B.GEMM_NO_ALLOC_SCRATCH_BYTES
    return A, Bm, to_device(A), to_device(Bm), p


def test_no_alloc_equals_gemm_run_on_two_calls():
    ensure_built()
    oracle.build()
    M, N, K, dtype = 300, 264, 2048, inputs.BF16
    A, Bm, dA, dB, p = _case(M, N, K, dtype, 0, 1, ("normal", 1.0), 4242, "streamk", tile_n=128)
    ref = run(p, dA, dB, M, N)                      # gemm_run, caller workspace
    C64, S, _ = oracle.gemm(A, Bm, M, N, K, dtype, 0, 1)
    ok, worst, nbad = oracle.check(ref, dtype, C64, S, K)
    assert ok, (nbad, worst)
    for _ in range(2):
        assert np.array_equal(_no_alloc(p, dA, dB, M, N), ref)
    p.close()


def test_no_alloc_integer_streamk_is_bit_exact():
    ensure_built()
    oracle.build()
    # every tile in the Stream-K wave: 5 x 4 tiles of 128 x 128 with 64
    # k-iterations each over all SMs, so every tile is split among several
    # CTAs, whose partials meet in the array
    M, N, K, dtype = 640, 512, 4096, inputs.F16
    A, Bm, dA, dB, p = _case(M, N, K, dtype, 0, 0, inputs.INT_LAW, 4343, "streamk",
                             sk_mode=1, tile_n=128, cluster_m=1)
    _, _, Cref = oracle.gemm(A, Bm, M, N, K, dtype, 0, 0, with_abs=False)
    ref = run(p, dA, dB, M, N)
    assert np.array_equal(ref, Cref)
    for _ in range(2):
        assert np.array_equal(_no_alloc(p, dA, dB, M, N), Cref)
    p.close()


def test_no_alloc_plans_with_different_flag_layouts_take_turns():
    """A hybrid Stream-K plan (flags per split tile, one partial slot per CTA)
    and a split-K plan (flags per tile, one slot per tile and part) share the
    array in alternation; each must still equal its gemm_run result."""
    ensure_built()
    law = inputs.INT_LAW
    M1, N1, K1 = 512, 768, 3072
    A1, B1, dA1, dB1, p1 = _case(M1, N1, K1, inputs.BF16, 0, 1, law, 11, "streamk", tile_n=128)
    M2, N2, K2 = 256, 384, 4096
    A2, B2, dA2, dB2, p2 = _case(M2, N2, K2, inputs.F16, 1, 0, law, 12, "splitk")
    assert p2.info("split_k") > 1
    r1, r2 = run(p1, dA1, dB1, M1, N1), run(p2, dA2, dB2, M2, N2)
    for _ in range(2):
        assert np.array_equal(_no_alloc(p1, dA1, dB1, M1, N1), r1)
        assert np.array_equal(_no_alloc(p2, dA2, dB2, M2, N2), r2)
    p1.close()
    p2.close()


def test_no_alloc_runs_plans_without_workspace():
    ensure_built()
    M, N, K, dtype = 256, 4096, 1024, inputs.F16
    A, Bm = inputs.operands(M, N, K, dtype, 0, 0, inputs.INT_LAW, inputs.INT_LAW, 4444)
    dA, dB = to_device(A), to_device(Bm)
    p = B.Plan(M, N, K, dtype, 0, 0, "persistent")
    assert p.workspace_size == 0
    ref = run(p, dA, dB, M, N)
    for _ in range(2):
        assert np.array_equal(_no_alloc(p, dA, dB, M, N), ref)
    p.close()


def test_no_alloc_rejects_oversized_workspace():
    ensure_built()
    M, N, K, dtype = 256, 4096, 1024, inputs.F16
    p = B.Plan(M, N, K, dtype, 0, 0, "streamk", tile_n=256)
    if p.workspace_size <= B.GEMM_NO_ALLOC_SCRATCH_BYTES:
        p.close()
        pytest.skip("this GPU's default grid fits the scratch array")
    buf = torch.zeros(max(M * K, K * N, M * N), dtype=torch.int16, device="cuda")
    with pytest.raises(B.GemmError) as e:
        B.gemm_run_no_alloc(p.handle, buf, buf, buf)
    assert e.value.status == B.GEMM_ERR_WORKSPACE
    p.close()
