"""GB300 (sm_103a) dense GEMM: C = A*B with fp16/bf16 inputs and fp32
accumulation, with data-parallel, persistent and Stream-K tile schedules.

The compute runs in ``libpsm_gemm.so`` (hand-written CUDA, C ABI in
include/gemm.h).  This package is its ctypes binding plus the seeded operand
generator.  Loading the binding's functions fails loudly if the library is
not built: there is no CPU fallback.
"""
from ._binding import (  # noqa: F401
    GEMM_BF16, GEMM_COL_MAJOR, GEMM_SCHED_AUTO, GEMM_F16, GEMM_ROW_MAJOR, GEMM_SCHED_DATA_PARALLEL,
    GEMM_SCHED_PERSISTENT, GEMM_SCHED_SPLITK, GEMM_SCHED_STREAMK, GemmError, Plan, SCHEDULES, gemm_last_status,
    gemm_plan_create, gemm_plan_create_offline, gemm_plan_destroy, gemm_plan_get_info,
    gemm_plan_set_option, gemm_plan_set_trace, gemm_plan_tile_coords, gemm_plan_units, gemm_run,
    gemm_run_host, gemm_run_no_alloc, gemm_status_string, gemm_workspace_size, load,
)
