/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Computes C = A * B with fp16 or bf16 inputs, fp32 accumulation and an
 * output of the input type, rounded once to nearest-even.  The output tiles
 * are scheduled three ways:
 *
 *   GEMM_SCHED_DATA_PARALLEL  one CTA per output tile, which ends after its
 *                             tile (HF post "naive vs persistent matmul":
 *                             the naive tiled matmul; GitHub issue
 *                             "Stream-k matmul implementation very slow ...",
 *                             final version, "tile matmul (grid=0)").
 *   GEMM_SCHED_PERSISTENT     one CTA per SM, each looping over tiles in a
 *                             grouped raster order (HF post: persistent
 *                             matmul; issue, final version, swizzle_tile).
 *   GEMM_SCHED_STREAMK        hybrid Stream-K (issue, final version, wrapper
 *                             and first_wave): the first sk tiles are split
 *                             evenly by k-iteration over g CTAs, the rest are
 *                             whole tiles.  Split tiles are fixed up through
 *                             a fp32 workspace and per-tile flags, in a fixed
 *                             order, so results are deterministic.
 *   GEMM_SCHED_SPLITK         fixed split-K (the issue's closing comments name
 *                             it as the alternative decomposition): every
 *                             tile's K range is cut into S near-equal parts
 *                             (GEMM_OPT_SPLIT_K), computed by a persistent
 *                             grid and fixed up like Stream-K.
 *   GEMM_SCHED_AUTO           the plan picks one of the above from the shape
 *                             (GEMM_INFO_SCHEDULE, GEMM_INFO_SK_MODE and
 *                             GEMM_INFO_SPLIT_K_CLUSTER report which): split-K
 *                             reduced inside clusters when it fits one wave
 *                             (for more than one row of 128-row tiles, only
 *                             with parts of at least 8 k-blocks); else
 *                             Stream-K for a single row of tiles;
 *                             persistent for tiny problems, for nearly one
 *                             full wave, and for 4+ waves of short tiles
 *                             (< 64 k-iterations, < 12 waves); Stream-K
 *                             (hybrid, or all tiles when the hybrid would
 *                             split a few tiles many ways) otherwise.
 *
 * Conventions for every entry point:
 *  - Each call returns a gemm_status_t; nothing else crosses the ABI.  An
 *    out-parameter is left untouched when the call fails.
 *  - Matrices are dense.  A is M x K, B is K x N, both row- or column-major
 *    (leading dimension K or M for A, N or K for B).  C is M x N row-major
 *    (leading dimension N).  Elements are 16-bit (fp16 or bf16, one type for
 *    A, B and C).
 *  - A, B, C and the workspace are DEVICE pointers owned by the caller, on the
 *    device that was current when the plan was created.  They must be 16-byte
 *    aligned.  K and N must be multiples of 8; M must be one too when A is
 *    column-major (the hardware tensor copy needs 16-byte row strides).
 *    Otherwise gemm_run returns GEMM_ERR_UNSUPPORTED.
 *  - gemm_run is asynchronous on the given stream.  Launch errors return at
 *    once; a device-side wait that ran out of time is reported by
 *    gemm_last_status.  Kernels are launched as programmatic dependents: a
 *    launch may begin while the previous kernel in the stream finishes, but
 *    it reads and writes global memory only after that kernel has completed.
 *  - A plan is not thread-safe.  Two runs that share one workspace must not
 *    overlap in time (use one stream or order them).
 */
#ifndef PSM_GEMM_H
#define PSM_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_F16 = 0, GEMM_BF16 = 1 } gemm_dtype_t;
typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;
typedef enum {
    GEMM_SCHED_DATA_PARALLEL = 0,
    GEMM_SCHED_PERSISTENT = 1,
    GEMM_SCHED_STREAMK = 2,
    GEMM_SCHED_SPLITK = 3,
    GEMM_SCHED_AUTO = 4
} gemm_schedule_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,  /* NULL handle/pointer, negative size, bad enum or key */
    GEMM_ERR_UNSUPPORTED = 2,  /* alignment / stride / option value not supported */
    GEMM_ERR_WORKSPACE = 3,    /* workspace NULL or misaligned while one is needed */
    GEMM_ERR_CUDA = 4,         /* a CUDA runtime call failed */
    GEMM_ERR_LAUNCH = 5,       /* the kernel launch was refused (e.g. grid not co-resident) */
    GEMM_ERR_TIMEOUT = 6,      /* a bounded device wait gave up; the tile's C was not written */
    GEMM_ERR_NO_DEVICE = 7     /* no CUDA device, or not an sm_103 device, or an offline plan */
} gemm_status_t;

/* cudaStream_t without the CUDA headers: the same type. NULL = default stream. */
typedef struct CUstream_st *gemm_stream_t;

typedef struct gemm_plan *gemm_plan_t;

/* Options for gemm_plan_set_option (key, value). */
enum {
    /* g: CTAs of the persistent / Stream-K grid. 0 (default) = number of SMs.
     * Must not exceed the SM count for GEMM_SCHED_STREAMK (the CTAs wait on
     * one another, so all must be resident at once). */
    GEMM_OPT_GRID = 1,
    /* rows of tiles per raster group (issue, final version, GROUP_M); 0 selects
     * the linear raster.  Default 8 for PERSISTENT and STREAMK, 0 for
     * DATA_PARALLEL. */
    GEMM_OPT_GROUP_M = 2,
    /* output tile width BN: 64, 128 or 256; 0 (default) lets the plan
     * choose.  The tile height is 128 rows and the k-slice 64.  64-wide tiles
     * run without clusters (GEMM_OPT_CLUSTER_M = 2 with them is UNSUPPORTED). */
    GEMM_OPT_TILE_N = 3,
    /* 1 (default): the issue's "two_tiles" rule adds g more Stream-K tiles
     * when more than g whole tiles would remain; 0: sk = tiles mod g. */
    GEMM_OPT_TWO_TILES = 4,
    /* bound on a Stream-K or split-K owner's wait for its peers, and on a
     * cluster split-K part's wait for the other parts of its tile,
     * microseconds (default 1000000).  On expiry the waiting CTA does not
     * write its part of C and gemm_last_status reports GEMM_ERR_TIMEOUT. */
    GEMM_OPT_WAIT_LIMIT_US = 5,
    /* test hook: the CTA with this index skips posting its peer flag, so its
     * owner's wait runs out (cluster split-K: it skips signalling the other
     * parts of its tile, whose waits run out).  -1 (default) = off. */
    GEMM_OPT_INJECT_SKIP_POST = 6,
    /* CTAs per cluster along M: 1, or 2 (two CTAs on adjacent 128-row halves
     * of a 256-row tile share one B tile, each loading half and multicasting
     * it to both).  0 (default) lets the plan choose (2 for wide tiles with at
     * least two row tiles).  With 2, the scheduler's tiles are 256 rows tall,
     * GEMM_OPT_GRID counts CTAs (pairs of them form one scheduling unit). */
    GEMM_OPT_CLUSTER_M = 7,
    /* Stream-K tile count: 0 (default) = the hybrid rule of the issue's final
     * version (tiles mod g, plus g under GEMM_OPT_TWO_TILES; the rest are whole
     * tiles); 1 = every tile goes to the Stream-K wave (the iteration space of
     * the whole product is split evenly over the g CTAs). */
    GEMM_OPT_SK_MODE = 8,
    /* split-K parts per tile for GEMM_SCHED_SPLITK; 0 (default) = as many
     * as fit in one round of the grid, floor(units / tiles), at least 1 and
     * at most ceil(K/64)/4.  With GEMM_OPT_SPLIT_K_CLUSTER: 2, 4 or 8, at
     * most ceil(K/64). */
    GEMM_OPT_SPLIT_K = 9,
    /* k order of whole tiles: 1 = tile t starts at k-block t*ipt/tiles and
     * wraps around (changes only the fp32 summation order of those tiles),
     * 0 (default) = ascending. */
    GEMM_OPT_K_ROTATE = 10,
    /* k-blocks of B prefetched into L2 ahead of the shared-memory ring
     * (0 = off, the default; up to 256). */
    GEMM_OPT_L2_PREFETCH = 11,
    /* with 2-CTA clusters: 1 (default) = one tcgen05 pair MMA (cta_group::2,
     * 256 x BN) per k-step issued for both CTAs, each CTA holding only its
     * half of B (deeper ring); 0 = each CTA runs its own 128 x BN MMA on a
     * full B tile assembled by TMA multicast. */
    GEMM_OPT_PAIR_MMA = 12,
    /* tile order: 0 (default) = the grouped raster of GEMM_OPT_GROUP_M (or
     * linear); 1 = along a Hilbert curve over the tile grid (the blog summary
     * "Inside NVIDIA GPUs: Anatomy of high performance matmul kernels" lists
     * Hilbert-curve scheduling).  The order is built on the host and copied
     * to a small device table owned by the plan when the option is set. */
    GEMM_OPT_RASTER = 13,
    /* gemm_run_host, row chunks of its block grid: 0 (default) = min(4,
     * M / 1024) when M and N are both >= 2048, min(8, M / 512) when only M is,
     * else 1; 1 = no row split; 2..16 = that many (each a whole number of
     * scheduled tile rows, so fewer may result).  The whole call is serial when
     * the grid has one block, or when the blocks' sub-plans would need more
     * workspace than gemm_workspace_size of this plan.  GEMM_INFO_HOST_CHUNKS
     * reports the count used. */
    GEMM_OPT_HOST_CHUNKS = 14,
    /* gemm_run_host, column chunks: 0 (default) = min(4, N / 1024) when M and
     * N are both >= 2048, min(8, N / 512) when only N is, else 1; 1 = no
     * column split; 2..16 = that many (whole tile columns).
     * GEMM_INFO_HOST_COL_CHUNKS reports the count used. */
    GEMM_OPT_HOST_COL_CHUNKS = 15,
    /* GEMM_SCHED_SPLITK only.  0 (default): the parts of a tile meet through
     * the workspace (fp32 partial slots and per-tile flags).  1: the S parts
     * of a tile run as one thread-block cluster of S CTAs (S = 2, 4 or 8,
     * GEMM_OPT_SPLIT_K; default the most that keep every tile in one wave),
     * and add their fp32 partials through distributed shared memory in
     * ascending k, so the plan needs no workspace; the sum order and so the
     * result bits are those of the workspace form with the same S.  Tiles
     * are 1-CTA (GEMM_OPT_CLUSTER_M = 2 and 64-wide tiles are UNSUPPORTED).
     * Unless GEMM_OPT_TILE_N or GEMM_OPT_SPLIT_K fix them, the tile width
     * (256 or 128) and S are the pair with the most CTAs in one wave of the
     * grid (GEMM_OPT_GRID, default #SMs) whose clusters can all be resident
     * at once, 256-wide tiles and then more parts first.  The grid is
     * tiles x S CTAs.  A split of K reduced inside a cluster has
     * no counterpart on the pages (the issue's closing comments name split-K
     * only). */
    GEMM_OPT_SPLIT_K_CLUSTER = 16,
    /* k-blocks of A and B of each CTA's first unit prefetched into L2 before
     * the launch waits for the previous kernel in the stream: 0 = off, up to
     * 256; -1 (default) = 8 when the launch fills at least three quarters of
     * the SMs, else 0 (GEMM_INFO_EARLY_PREFETCH reports the value used).  A CTA
     * that starts while the previous kernel drains uses that kernel's tail to
     * fetch its first operands.  Only L2 is filled (the point of coherence),
     * so results are unchanged whatever the previous kernel wrote.  No
     * counterpart on the pages. */
    GEMM_OPT_EARLY_PREFETCH = 17
};

/* Keys for gemm_plan_get_info. */
enum {
    GEMM_INFO_TILE_M = 1,           /* rows of a scheduled tile: 128 x cluster size */
    GEMM_INFO_TILE_N = 2, GEMM_INFO_TILE_K = 3,
    GEMM_INFO_TILES_M = 4, GEMM_INFO_TILES_N = 5, GEMM_INFO_TILES = 6,
    GEMM_INFO_ITERS_PER_TILE = 7,   /* k-iterations per tile, ceil(K / 64) */
    GEMM_INFO_GRID = 8,             /* CTAs launched by gemm_run */
    GEMM_INFO_SK_TILES = 9,         /* tiles split by the Stream-K wave */
    GEMM_INFO_SK_ITERS_PER_CTA = 10,/* even share of Stream-K iterations */
    GEMM_INFO_SK_ITERS_REM = 11,    /* CTAs that take one iteration more */
    GEMM_INFO_NUM_SMS = 12,
    GEMM_INFO_STAGES = 13,          /* depth of the shared-memory ring */
    GEMM_INFO_GROUP_M = 14,
    GEMM_INFO_SMEM_BYTES = 15,      /* dynamic shared memory per CTA */
    GEMM_INFO_CLUSTER_M = 16,       /* CTAs per cluster (1 or 2) */
    GEMM_INFO_A_ROWS_PER_STAGE = 17,/* rows of A each ring stage loads: 128, or 64 when M <= 64 */
    GEMM_INFO_SPLIT_K = 18,         /* split-K parts per tile (0 unless GEMM_SCHED_SPLITK;
                                       with GEMM_OPT_SPLIT_K_CLUSTER, the cluster size) */
    GEMM_INFO_K_ROTATE = 19,        /* 1 when whole tiles rotate their k order */
    GEMM_INFO_L2_PREFETCH = 20,     /* k-blocks of B prefetched into L2 ahead of the ring */
    GEMM_INFO_PAIR_MMA = 21,        /* 1 when the cluster runs pair MMAs */
    GEMM_INFO_SCHEDULE = 22,        /* the schedule that runs (GEMM_SCHED_AUTO resolved) */
    GEMM_INFO_SK_MODE = 23,         /* 1 when every tile is in the Stream-K wave */
    GEMM_INFO_RASTER = 24,          /* 0 grouped / linear, 1 Hilbert */
    GEMM_INFO_HOST_CHUNKS = 25,     /* row chunks of gemm_run_host's block grid */
    GEMM_INFO_HOST_COL_CHUNKS = 26, /* column chunks (both 1: serial) */
    GEMM_INFO_SPLIT_K_CLUSTER = 27, /* 1 when split-K parts reduce inside a cluster */
    GEMM_INFO_CLUSTERS_RESIDENT = 28,/* clusters of this plan's kernel that fit the GPU at
                                        once (0: no clusters, or an offline plan) */
    GEMM_INFO_EARLY_PREFETCH = 29   /* k-blocks prefetched into L2 before the grid wait */
};

/* Roles of a work unit reported by gemm_plan_units.  CLUSTER_PART: one k-part
 * of a tile under GEMM_OPT_SPLIT_K_CLUSTER, reduced with the other parts of
 * its cluster. */
enum { GEMM_ROLE_FULL = 0, GEMM_ROLE_OWNER = 1, GEMM_ROLE_PEER = 2, GEMM_ROLE_CLUSTER_PART = 3 };

/*
 * Create a plan for one problem shape on the current CUDA device.
 * Tile grid and Stream-K split: issue, final version, wrapper (_call).
 * M, N, K >= 0.  *out receives a handle that gemm_plan_destroy frees.
 * Errors: INVALID_ARG (NULL out, negative size, bad enum), NO_DEVICE (no
 * device, or the device is not compute capability 10.3), CUDA.
 */
gemm_status_t gemm_plan_create(gemm_plan_t *out, int64_t M, int64_t N, int64_t K,
                               gemm_dtype_t dtype, gemm_layout_t layout_a,
                               gemm_layout_t layout_b, gemm_schedule_t schedule);

/*
 * Same as gemm_plan_create but touches no device: a plan for inspection only
 * (gemm_plan_get_info, gemm_plan_units, gemm_workspace_size) as if the device
 * had num_sms SMs.  gemm_run on it returns GEMM_ERR_NO_DEVICE.  The pages
 * have no counterpart (their wrapper derives the split at launch time).
 * Errors: INVALID_ARG (as gemm_plan_create, or num_sms <= 0).
 */
gemm_status_t gemm_plan_create_offline(gemm_plan_t *out, int64_t M, int64_t N, int64_t K,
                                       gemm_dtype_t dtype, gemm_layout_t layout_a,
                                       gemm_layout_t layout_b, gemm_schedule_t schedule,
                                       int num_sms);

/* Set one GEMM_OPT_* option; the plan is re-derived.  The tuning options
 * stand for the launch parameters of the issue's final version, matmul.apply
 * (grid, block sizes, two_tiles) and the GROUP_M of swizzle_tile; the others
 * (clusters, split-K parts, raster, host chunks, test hooks) have no
 * counterpart on the pages.  On error the plan keeps its previous options.
 * Errors: INVALID_ARG (NULL plan, unknown key), UNSUPPORTED (value out of
 * range). */
gemm_status_t gemm_plan_set_option(gemm_plan_t plan, int key, int64_t value);

/* Read one GEMM_INFO_* value into *value.  The derived counts (tiles,
 * iterations per tile, Stream-K tiles, the even split) are those the issue's
 * final version computes in its wrapper (_call); the rest have no counterpart
 * on the pages.  Errors: INVALID_ARG (NULL plan or value, unknown key). */
gemm_status_t gemm_plan_get_info(gemm_plan_t plan, int key, int64_t *value);

/*
 * Bytes of device workspace gemm_run needs: 0 for DATA_PARALLEL and
 * PERSISTENT; for STREAMK, 8 bytes of flag per split tile and cluster half
 * (rounded up to 256) plus one 128 x BN fp32 partial-tile slot per CTA (the
 * "scratchpad" of the Stream-K fixup mentioned in the issue, second code
 * version); for SPLITK, a flag per tile and half plus a slot per tile, part
 * beyond the first, and half.
 * The caller allocates it (16-byte aligned) and owns it; the plan clears the
 * flag part the first time it sees a workspace address.  Errors: INVALID_ARG.
 */
gemm_status_t gemm_workspace_size(gemm_plan_t plan, size_t *bytes);

/*
 * C = A * B on `stream`, asynchronously: one kernel launch.  Counterpart of
 * the issue's final version, matmul.apply / _call, which launches the
 * Stream-K kernel (first_wave) and then the whole-tile kernel (full_tiles);
 * here one persistent launch runs both parts.  `workspace` may be NULL only
 * when gemm_workspace_size is 0.  C is written in full (every element, once);
 * A and B are only read.  M == 0 or N == 0: nothing is done.  K == 0: C is
 * set to +0.
 * Errors: INVALID_ARG (NULL plan or operand), UNSUPPORTED (alignment),
 * WORKSPACE, NO_DEVICE (offline plan), CUDA, LAUNCH.
 */
gemm_status_t gemm_run(gemm_plan_t plan, const void *A, const void *B, void *C,
                       void *workspace, gemm_stream_t stream);

/*
 * End-to-end variant (the pages time the device only and have no
 * counterpart): copies hA -> dA and hB -> dB (host to device), runs
 * C = A * B on the device copies, and copies dC -> hC (device to host).  All
 * six buffers are the caller's, in the layouts of the plan; host buffers
 * should be pinned for the copies to be asynchronous.
 *  - Serial (a one-block grid, see GEMM_OPT_HOST_CHUNKS and
 *    GEMM_OPT_HOST_COL_CHUNKS): the three steps are enqueued on `stream`, the
 *    product through gemm_run.
 *  - Pipelined over an nr x nc grid of blocks: row chunks of A and column
 *    chunks of B are copied in on an internal stream (A_0, B_0, A_1, B_1,
 *    ...); block (i, j) of C is computed on `stream` once A_i and B_j have
 *    arrived and copied out on a second internal stream, so copies and
 *    compute overlap.  The call
 *    records an event on `stream` before its first copy and makes `stream`
 *    wait for the last copy out, so everything enqueued on `stream` before
 *    the call precedes it and everything after it follows it.  The first
 *    pipelined call of a plan creates the two streams, the events and two
 *    internal sub-plans (released by gemm_plan_destroy or an option change;
 *    if they cannot be made, the call runs the serial path instead);
 *    the chunks run one after another on `stream` and share `workspace`.
 * Errors: as gemm_run; CUDA when a copy, stream or event call fails.
 */
gemm_status_t gemm_run_host(gemm_plan_t plan, const void *hA, const void *hB, void *hC,
                            void *dA, void *dB, void *dC, void *workspace,
                            gemm_stream_t stream);

/* Size of the fixed scratch array behind gemm_run_no_alloc: 16 MiB. */
#define GEMM_NO_ALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * Same product as gemm_run, for callers that cannot allocate device memory
 * (for example a plug-in inside a framework that owns all device memory and
 * forbids allocation on its execution path).  The pages have no counterpart:
 * this is a library convenience.  The caller passes A, B and C as for
 * gemm_run but no workspace: the Stream-K flags and partial tiles go to a
 * fixed 16 MiB device array inside the library, which each GPU that loads the
 * library holds until the process exits.  Nothing is allocated by this call
 * (no cudaMalloc, cudaFree or allocating library routine).
 *  - Plans whose gemm_workspace_size exceeds GEMM_NO_ALLOC_SCRATCH_BYTES are
 *    rejected with GEMM_ERR_WORKSPACE (choose GEMM_OPT_TILE_N = 128 or a
 *    smaller GEMM_OPT_GRID to fit).  Plans that need no workspace just run.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call shares the one array and finds the last call's data in it;
 *    each call clears the flag part on `stream` before its kernel.  Calls
 *    that overlap on the GPU (other streams, other threads) race: serialise
 *    them.
 * Errors: as gemm_run, plus WORKSPACE as above.
 */
gemm_status_t gemm_run_no_alloc(gemm_plan_t plan, const void *A, const void *B, void *C,
                                gemm_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the plan's device status word.
 * Returns GEMM_OK, GEMM_ERR_TIMEOUT (a bounded device wait expired since the
 * last call), or GEMM_ERR_CUDA (the stream reported an error).  The pages
 * have no counterpart: the spin lock of the issue's fixup waits without a
 * bound and reports nothing.  Errors: INVALID_ARG (NULL plan), NO_DEVICE
 * (offline plan).
 */
gemm_status_t gemm_last_status(gemm_plan_t plan, gemm_stream_t stream);

/*
 * Host twin of the device tile scheduler: the work units CTA `cta` executes,
 * in order (the two CTAs of a cluster execute the same units, each on its
 * 128-row half of the GEMM_INFO_TILE_M-row tile), 5 int32 per unit: tile id
 * (raster order), first k-iteration,
 * end k-iteration, role (GEMM_ROLE_*), peers (for an OWNER: how many peer
 * partials it adds; else 0).  Writes at most max_units units to `units`
 * (may be NULL when max_units is 0) and the full count to *n_units.  For a
 * CLUSTER_PART unit, peers holds the number of other parts of its tile.
 * Segments: issue, final version, first_wave (the range of a program cut at
 * tile boundaries) and full_tiles.  Errors: INVALID_ARG.
 */
gemm_status_t gemm_plan_units(gemm_plan_t plan, int64_t cta, int32_t *units,
                              int64_t max_units, int64_t *n_units);

/*
 * Measurement hook (no counterpart on the pages, which time whole launches
 * only): when `device_buffer` is not NULL, every later gemm_run of
 * this plan writes six uint64 stamps per CTA into it: four %globaltimer
 * stamps (nanoseconds) at CTA start, prologue done, last operand copy
 * issued and CTA end, then the SM's %clock64 (cycles) at CTA start and end,
 * whose ratio to the elapsed nanoseconds is the SM clock the CTA ran at; CTA
 * c at index 6*c.  It must hold at least 6 * 8 * GEMM_INFO_GRID bytes, else
 * no stamps are written.  The caller owns the buffer.  NULL turns stamps off.
 * Used to measure the idle time of SMs at the wave tail of each schedule.
 * Errors: INVALID_ARG (NULL plan or a buffer not 8-byte aligned).
 */
gemm_status_t gemm_plan_set_trace(gemm_plan_t plan, void *device_buffer, size_t bytes);

/* Tile coordinates (tile row, tile column) of raster id `tile` (issue, final
 * version, swizzle_tile / linear_tile).  Errors: INVALID_ARG. */
gemm_status_t gemm_plan_tile_coords(gemm_plan_t plan, int64_t tile, int64_t *tile_m,
                                    int64_t *tile_n);

/* Free the plan, its device status word, its raster table and the
 * gemm_run_host pipeline (streams, events, sub-plans).  NULL is accepted.
 * The pages have no counterpart (the Python wrapper frees nothing
 * explicitly).  Always returns GEMM_OK. */
gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* Static text for a status code (never NULL; unknown codes give
 * "GEMM_ERR_UNKNOWN").  The pages have no counterpart: their error handling
 * is assertions. */
const char *gemm_status_string(gemm_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* PSM_GEMM_H */
