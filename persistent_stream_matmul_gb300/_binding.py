"""ctypes binding of the C ABI in include/gemm.h.

Argument marshalling only: every step of the product runs in the CUDA
library.  The functions keep the C names; a non-OK status raises GemmError.
Device operands may be given as integers (device addresses) or as objects
with a ``data_ptr()`` method (torch tensors); streams as integers or objects
with a ``cuda_stream`` attribute.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpsm_gemm.so")

GEMM_F16, GEMM_BF16 = 0, 1
GEMM_ROW_MAJOR, GEMM_COL_MAJOR = 0, 1
GEMM_SCHED_DATA_PARALLEL, GEMM_SCHED_PERSISTENT, GEMM_SCHED_STREAMK, GEMM_SCHED_SPLITK = 0, 1, 2, 3
GEMM_SCHED_AUTO = 4
SCHEDULES = {"dp": 0, "persistent": 1, "streamk": 2, "splitk": 3, "auto": 4}

(GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_WORKSPACE, GEMM_ERR_CUDA,
 GEMM_ERR_LAUNCH, GEMM_ERR_TIMEOUT, GEMM_ERR_NO_DEVICE) = range(8)

GEMM_OPT_GRID = 1
GEMM_OPT_GROUP_M = 2
GEMM_OPT_TILE_N = 3
GEMM_OPT_TWO_TILES = 4
GEMM_OPT_WAIT_LIMIT_US = 5
GEMM_OPT_INJECT_SKIP_POST = 6
GEMM_OPT_CLUSTER_M = 7
GEMM_OPT_SK_MODE = 8
GEMM_OPT_SPLIT_K = 9
GEMM_OPT_K_ROTATE = 10
GEMM_OPT_L2_PREFETCH = 11
GEMM_OPT_PAIR_MMA = 12
GEMM_OPT_RASTER = 13
GEMM_OPT_HOST_CHUNKS = 14
GEMM_OPT_HOST_COL_CHUNKS = 15
GEMM_OPT_SPLIT_K_CLUSTER = 16
GEMM_OPT_EARLY_PREFETCH = 17

INFO = {
    "tile_m": 1, "tile_n": 2, "tile_k": 3, "tiles_m": 4, "tiles_n": 5, "tiles": 6,
    "iters_per_tile": 7, "grid": 8, "sk_tiles": 9, "sk_iters_per_cta": 10,
    "sk_iters_rem": 11, "num_sms": 12, "stages": 13, "group_m": 14, "smem_bytes": 15, "cluster_m": 16,
    "a_rows_per_stage": 17, "split_k": 18, "k_rotate": 19,
    "l2_prefetch": 20, "pair_mma": 21, "schedule": 22, "sk_mode": 23, "raster": 24, "host_chunks": 25, "host_col_chunks": 26,
    "split_k_cluster": 27, "clusters_resident": 28, "early_prefetch": 29,
}
ROLE_FULL, ROLE_OWNER, ROLE_PEER, ROLE_CLUSTER_PART = 0, 1, 2, 3
TRACE_STAMPS = 6   # uint64 per CTA written by gemm_plan_set_trace: 4 timer + 2 clock stamps

# every entry point of include/gemm.h: name -> (restype, argtypes)
_i64, _i32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
_pp = ctypes.POINTER(ctypes.c_void_p)
SIGNATURES = {
    "gemm_plan_create": (_i32, [_pp, _i64, _i64, _i64, _i32, _i32, _i32, _i32]),
    "gemm_plan_create_offline": (_i32, [_pp, _i64, _i64, _i64, _i32, _i32, _i32, _i32, _i32]),
    "gemm_plan_set_option": (_i32, [_vp, _i32, _i64]),
    "gemm_plan_get_info": (_i32, [_vp, _i32, ctypes.POINTER(_i64)]),
    "gemm_workspace_size": (_i32, [_vp, ctypes.POINTER(ctypes.c_size_t)]),
    "gemm_run": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "gemm_run_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "gemm_last_status": (_i32, [_vp, _vp]),
    "gemm_run_no_alloc": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "gemm_plan_units": (_i32, [_vp, _i64, ctypes.POINTER(ctypes.c_int32), _i64,
                               ctypes.POINTER(_i64)]),
    "gemm_plan_tile_coords": (_i32, [_vp, _i64, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    "gemm_plan_set_trace": (_i32, [_vp, _vp, ctypes.c_size_t]),
    "gemm_plan_destroy": (_i32, [_vp]),
    "gemm_status_string": (ctypes.c_char_p, [_i32]),
}

_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s" % (where, gemm_status_string(status)))


def load(path: str = LIB_PATH):
    """Load the CUDA library; raise if it is missing (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(
                "libpsm_gemm.so is not built (%s); run persistent_stream_matmul_gb300.build.build()"
                % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(st: int, where: str):
    if st != GEMM_OK:
        raise GemmError(st, where)


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def gemm_plan_create(M, N, K, dtype, layout_a, layout_b, schedule) -> int:
    h = ctypes.c_void_p()
    _check(load().gemm_plan_create(ctypes.byref(h), M, N, K, dtype, layout_a, layout_b, schedule),
           "gemm_plan_create")
    return h.value


def gemm_plan_create_offline(M, N, K, dtype, layout_a, layout_b, schedule, num_sms) -> int:
    h = ctypes.c_void_p()
    _check(load().gemm_plan_create_offline(ctypes.byref(h), M, N, K, dtype, layout_a, layout_b,
                                           schedule, num_sms), "gemm_plan_create_offline")
    return h.value


def gemm_plan_set_option(plan, key, value):
    _check(load().gemm_plan_set_option(plan, key, value), "gemm_plan_set_option")


def gemm_plan_get_info(plan, key) -> int:
    v = ctypes.c_int64()
    key = INFO[key] if isinstance(key, str) else key
    _check(load().gemm_plan_get_info(plan, key, ctypes.byref(v)), "gemm_plan_get_info")
    return v.value


def gemm_workspace_size(plan) -> int:
    v = ctypes.c_size_t()
    _check(load().gemm_workspace_size(plan, ctypes.byref(v)), "gemm_workspace_size")
    return v.value


def gemm_run(plan, A, B, C, workspace=None, stream=None):
    _check(load().gemm_run(plan, _addr(A), _addr(B), _addr(C), _addr(workspace), _stream(stream)),
           "gemm_run")


def gemm_run_host(plan, hA, hB, hC, dA, dB, dC, workspace=None, stream=None):
    _check(load().gemm_run_host(plan, _addr(hA), _addr(hB), _addr(hC), _addr(dA), _addr(dB),
                                _addr(dC), _addr(workspace), _stream(stream)), "gemm_run_host")


def gemm_run_no_alloc(plan, A, B, C, stream=None):
    """gemm_run without a workspace argument: the library's fixed scratch array
    is used instead, so nothing is allocated (for callers that cannot allocate)."""
    _check(load().gemm_run_no_alloc(plan, _addr(A), _addr(B), _addr(C), _stream(stream)),
           "gemm_run_no_alloc")


GEMM_NO_ALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def gemm_last_status(plan, stream=None) -> int:
    """Returns the status code (GEMM_OK or GEMM_ERR_TIMEOUT ...); does not raise."""
    return int(load().gemm_last_status(plan, _stream(stream)))


def gemm_plan_units(plan, cta: int):
    """[(tile, k0, k1, role, npeers), ...] of CTA ``cta``."""
    n = ctypes.c_int64()
    _check(load().gemm_plan_units(plan, cta, None, 0, ctypes.byref(n)), "gemm_plan_units")
    buf = (ctypes.c_int32 * (5 * max(n.value, 1)))()
    _check(load().gemm_plan_units(plan, cta, buf, n.value, ctypes.byref(n)), "gemm_plan_units")
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(n.value)]


def gemm_plan_tile_coords(plan, tile: int):
    tm, tn = ctypes.c_int64(), ctypes.c_int64()
    _check(load().gemm_plan_tile_coords(plan, tile, ctypes.byref(tm), ctypes.byref(tn)),
           "gemm_plan_tile_coords")
    return tm.value, tn.value


def gemm_plan_set_trace(plan, device_buffer, nbytes: int):
    """Per-CTA stamps into a device buffer: %globaltimer at start, ready,
    loads done and end, then %clock64 at start and end (TRACE_STAMPS each)."""
    _check(load().gemm_plan_set_trace(plan, _addr(device_buffer), nbytes), "gemm_plan_set_trace")


def gemm_plan_destroy(plan):
    _check(load().gemm_plan_destroy(plan), "gemm_plan_destroy")


class Plan:
    """Owning wrapper around a plan handle (marshalling only)."""

    def __init__(self, M, N, K, dtype, layout_a, layout_b, schedule, offline_sms=None,
                 **options):
        if isinstance(schedule, str):
            schedule = SCHEDULES[schedule]
        self.M, self.N, self.K = M, N, K
        self.dtype, self.layout_a, self.layout_b, self.schedule = dtype, layout_a, layout_b, schedule
        if offline_sms is None:
            self.handle = gemm_plan_create(M, N, K, dtype, layout_a, layout_b, schedule)
        else:
            self.handle = gemm_plan_create_offline(M, N, K, dtype, layout_a, layout_b, schedule,
                                                   offline_sms)
        keys = {"grid": GEMM_OPT_GRID, "group_m": GEMM_OPT_GROUP_M, "tile_n": GEMM_OPT_TILE_N,
                "two_tiles": GEMM_OPT_TWO_TILES, "wait_limit_us": GEMM_OPT_WAIT_LIMIT_US,
                "inject_skip_post": GEMM_OPT_INJECT_SKIP_POST, "cluster_m": GEMM_OPT_CLUSTER_M,
                "sk_mode": GEMM_OPT_SK_MODE, "split_k": GEMM_OPT_SPLIT_K,
                "k_rotate": GEMM_OPT_K_ROTATE, "l2_prefetch": GEMM_OPT_L2_PREFETCH,
                "pair_mma": GEMM_OPT_PAIR_MMA, "raster": GEMM_OPT_RASTER,
                "host_chunks": GEMM_OPT_HOST_CHUNKS, "host_col_chunks": GEMM_OPT_HOST_COL_CHUNKS,
                "split_cluster": GEMM_OPT_SPLIT_K_CLUSTER, "early_prefetch": GEMM_OPT_EARLY_PREFETCH}
        for k, v in options.items():
            if v is not None:
                gemm_plan_set_option(self.handle, keys[k], int(v))

    def info(self, key):
        return gemm_plan_get_info(self.handle, key)

    def set_option(self, key, value):
        gemm_plan_set_option(self.handle, key, value)

    @property
    def workspace_size(self) -> int:
        return gemm_workspace_size(self.handle)

    def units(self, cta):
        return gemm_plan_units(self.handle, cta)

    def tile_coords(self, tile):
        return gemm_plan_tile_coords(self.handle, tile)

    def run(self, A, B, C, workspace=None, stream=None):
        gemm_run(self.handle, A, B, C, workspace, stream)

    def run_host(self, hA, hB, hC, dA, dB, dC, workspace=None, stream=None):
        gemm_run_host(self.handle, hA, hB, hC, dA, dB, dC, workspace, stream)

    def set_trace(self, device_buffer, nbytes):
        gemm_plan_set_trace(self.handle, device_buffer, nbytes)

    def last_status(self, stream=None) -> int:
        return gemm_last_status(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
