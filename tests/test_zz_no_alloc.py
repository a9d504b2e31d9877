"""gemm_run_no_alloc: the entry point for callers that cannot allocate device
memory (e.g. a plug-in inside a framework that owns all device memory).  It
keeps the Stream-K scratch in the library's fixed device array instead of a
caller workspace.  Its output must agree with gemm_run's within the tests'
acceptance bound, on two calls in a row.  This file is collected last."""
import numpy as np
import pytest
import torch

import oracle
from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import inputs
from tests.gpu_util import GUARD, SENTINEL, ensure_built, run, to_device

pytestmark = pytest.mark.gpu


def _no_alloc(plan, dA, dB, M, N):
    Cbuf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    B.gemm_run_no_alloc(plan.handle, dA, dB, Cbuf.data_ptr() + 2 * GUARD)
    assert plan.last_status() == B.GEMM_OK
    host = Cbuf.cpu().numpy().view(np.uint16)
    assert (host[:GUARD] == SENTINEL).all() and (host[-GUARD:] == SENTINEL).all()
    return host[GUARD:GUARD + M * N].reshape(M, N).copy()


def test_no_alloc_agrees_with_gemm_run_on_two_calls():
    ensure_built()
    oracle.build()
    M, N, K, dtype = 300, 264, 2048, inputs.BF16
    A, Bm = inputs.operands(M, N, K, dtype, 0, 1, ("normal", 1.0), ("normal", 1.0), 4242)
    dA, dB = to_device(A), to_device(Bm)
    p = B.Plan(M, N, K, dtype, 0, 1, "streamk", tile_n=128)
    assert 0 < p.workspace_size <= B.GEMM_NO_ALLOC_SCRATCH_BYTES
    ref = run(p, dA, dB, M, N)                      # gemm_run, caller workspace
    C64, S, _ = oracle.gemm(A, Bm, M, N, K, dtype, 0, 1)
    ref64 = oracle.decode(ref, dtype)
    bound = oracle.tolerance_bound(ref64, S, K)
    for _ in range(2):
        got = _no_alloc(p, dA, dB, M, N)
        assert np.all(np.abs(oracle.decode(got, dtype) - ref64) <= bound)
        ok, worst, nbad = oracle.check(got, dtype, C64, S, K)
        assert ok, (nbad, worst)
    p.close()


def test_no_alloc_rejects_oversized_workspace_and_runs_without_one():
    ensure_built()
    M, N, K, dtype = 256, 4096, 1024, inputs.F16
    p = B.Plan(M, N, K, dtype, 0, 0, "streamk", tile_n=256)
    if p.workspace_size <= B.GEMM_NO_ALLOC_SCRATCH_BYTES:
        pytest.skip("this GPU's default grid fits the scratch array")
    buf = torch.zeros(max(M * K, K * N, M * N), dtype=torch.int16, device="cuda")
    with pytest.raises(B.GemmError) as e:
        B.gemm_run_no_alloc(p.handle, buf, buf, buf)
    assert e.value.status == B.GEMM_ERR_WORKSPACE
    p.close()
    A, Bm = inputs.operands(M, N, K, dtype, 0, 0, inputs.INT_LAW, inputs.INT_LAW, 4343)
    dA, dB = to_device(A), to_device(Bm)
    p = B.Plan(M, N, K, dtype, 0, 0, "persistent")
    assert p.workspace_size == 0
    got = _no_alloc(p, dA, dB, M, N)
    assert np.array_equal(got, run(p, dA, dB, M, N))
    p.close()
