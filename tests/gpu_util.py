"""Helpers shared by the GPU tests: run the CUDA library through its C ABI on
seeded operands, with guard bands around C."""
import numpy as np
import torch

from persistent_stream_matmul_gb300 import _binding as B
from persistent_stream_matmul_gb300 import build

GUARD = 64               # elements of sentinel before and after C (multiple of 8)
SENTINEL = 0x7E5A        # a NaN pattern in both 16-bit types


def ensure_built():
    build.build()
    B.load()


def to_device(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda")


class Workspace:
    """Device workspace owned by the test (the caller owns it in the ABI)."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        return self.buf


def run(plan: B.Plan, dA: torch.Tensor, dB: torch.Tensor, M: int, N: int, ws: Workspace = None,
        stream=None, check_guard=True):
    """C = A*B on the GPU; returns C as uint16 (M, N) numpy, guards verified."""
    ws = ws or Workspace()
    Cbuf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    cptr = Cbuf.data_ptr() + 2 * GUARD
    w = ws.get(plan.workspace_size)
    plan.run(dA, dB, cptr, w, stream)
    st = plan.last_status(stream)
    if st != B.GEMM_OK:
        raise B.GemmError(st, "gemm_last_status")
    host = Cbuf.cpu().numpy().view(np.uint16)
    if check_guard:
        assert (host[:GUARD] == SENTINEL).all() and (host[-GUARD:] == SENTINEL).all(), \
            "write outside C"
    return host[GUARD:GUARD + M * N].reshape(M, N).copy()
