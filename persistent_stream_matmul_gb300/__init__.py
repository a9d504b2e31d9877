"""GB300 (sm_103a) dense GEMM with data-parallel, persistent and Stream-K tile schedules."""
