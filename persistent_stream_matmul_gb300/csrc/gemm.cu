// Host side of the GEMM library: plans, tensor-map encoding, launches and the
// C ABI declared in include/gemm.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <vector>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm.h"
#include "gemm_kernel.cuh"

using namespace psm;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Run numbers tagged into the Stream-K flags.  Global so that plans sharing
// one workspace never reuse a number; 0 is never handed out, so a zeroed flag
// matches no run.
std::atomic<uint32_t> g_epoch{0x1000u};

uint32_t next_epoch() {
    uint32_t e;
    do { e = ++g_epoch; } while (e == 0);
    return e;
}

int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Cell d of the Hilbert curve over a side x side square (side a power of
// two), as (x, y): the classic index-to-coordinates walk, which at each scale
// picks the quadrant from two bits of d and rotates / reflects the lower
// levels into it.
void hilbert_cell(int64_t side, int64_t d, int64_t& x, int64_t& y) {
    x = y = 0;
    for (int64_t sz = 1; sz < side; sz *= 2) {
        const int64_t rx = 1 & (d / 2);
        const int64_t ry = 1 & (d ^ rx);
        if (ry == 0) {
            if (rx == 1) {
                x = sz - 1 - x;
                y = sz - 1 - y;
            }
            const int64_t t = x;
            x = y;
            y = t;
        }
        x += sz * rx;
        y += sz * ry;
        d /= 4;
    }
}

// Tile order along the Hilbert curve of the smallest power-of-two square
// that covers the tile grid, keeping the cells inside it.
void hilbert_order(int64_t tiles_m, int64_t tiles_n, std::vector<int32_t>& out) {
    int64_t side = 1;
    while (side < tiles_m || side < tiles_n) side *= 2;
    out.clear();
    out.reserve((size_t)(tiles_m * tiles_n));
    for (int64_t d = 0; d < side * side; ++d) {
        int64_t x, y;
        hilbert_cell(side, d, x, y);
        if (y < tiles_m && x < tiles_n) out.push_back((int32_t)((y << 16) | x));
    }
}

}  // namespace

struct gemm_plan {
    int64_t M, N, K;
    int dtype, layout_a, layout_b, schedule;
    int device, num_sms, offline;
    // options
    int opt_grid, opt_group_m, opt_tile_n, opt_two_tiles, inject_skip, opt_cluster_m, opt_sk_mode;
    int opt_split, opt_k_rotate, opt_l2_prefetch, opt_pair_mma;
    int opt_split_cluster;  // GEMM_SCHED_SPLITK: 1 = parts reduce inside a cluster
    int opt_early_prefetch; // k-blocks of the first unit prefetched into L2 before the grid wait
    int eff_schedule;  // the schedule that runs (GEMM_SCHED_AUTO resolved)
    int eff_sk_mode;   // its Stream-K mode (GEMM_SCHED_AUTO resolved)
    int opt_raster;    // 0: grouped / linear (GROUP_M), 1: Hilbert curve
    std::vector<int32_t>* raster_host;  // Hilbert order, (row << 16) | column
    int32_t* raster_dev;                // device copy
    int64_t raster_tiles;               // entries in both
    int64_t wait_limit_us;
    int64_t a_ld;         // leading dimension of a column-major A in elements (0: M)
    int64_t b_ld;         // leading dimension of a row-major B in elements (0: N)
    int64_t c_ld;         // leading dimension of C in elements (0: N)
    int opt_host_chunks;      // gemm_run_host row chunks: 0 auto, 1 none, 2..16
    int opt_host_col_chunks;  // gemm_run_host column chunks: 0 auto, 1 none, 2..16
    // gemm_run_host pipeline, made on its first pipelined call
    gemm_plan* sub[4];    // sub-plans: [last row chunk?][last column chunk?]
    int64_t sub_rows, sub_cols;  // rows and columns of a full block
    cudaStream_t h2d, d2h;
    cudaEvent_t ev_start, ev_done, ev_a[16], ev_b[16], ev_c[64];
    bool pipe_ready;
    bool owns_status;     // false for a sub-plan: it reports into its parent's word
    int max_pair_ctas;  // CTAs co-resident as 2-CTA clusters (0: unknown)
    // derived
    int BN, CM, AROWS, PAIR, ctas, stages, smem_bytes;
    Sched s;
    size_t ws_flag_bytes, ws_bytes;
    // device state
    int* d_status;
    // caches
    const void* tm_a_ptr;
    const void* tm_b_ptr;
    bool tm_valid;
    CUtensorMap tmA, tmB;
    // C's tensor map (pair-MMA kernels): for this pointer and row stride;
    // state 0 unknown, 1 usable, -1 not usable (alignment)
    const void* tm_c_ptr;
    int64_t tm_c_ld;
    int tm_c_state;
    CUtensorMap tmC;
    const void* flags_cleared_for;
    bool attr_set[40];
    unsigned long long* trace;  // optional per-CTA stamps (caller-owned device buffer)
    size_t trace_bytes;
};

namespace {

bool valid_enums(int dtype, int la, int lb, int sched) {
    return (dtype == GEMM_F16 || dtype == GEMM_BF16) && (la == 0 || la == 1) &&
           (lb == 0 || lb == 1) && (sched >= 0 && sched <= 4);
}

template <int BN, bool BF, int CM, int AROWS = 128, bool PAIR_MMA = false, bool KCL = false>
void* kernel_ptr() {
    return reinterpret_cast<void*>(&gemm_kernel<BN, BF, CM, AROWS, PAIR_MMA, KCL>);
}

// cluster split-K kernels: 1-CTA MMAs, BN = 128 or 256, AROWS = 128 or 64
void* pick_kernel_kcl(int BN, int dtype, int AROWS) {
    const bool bf = dtype == GEMM_BF16;
    if (BN == 256) {
        if (AROWS == 64)
            return bf ? kernel_ptr<256, true, 1, 64, false, true>() : kernel_ptr<256, false, 1, 64, false, true>();
        return bf ? kernel_ptr<256, true, 1, 128, false, true>() : kernel_ptr<256, false, 1, 128, false, true>();
    }
    if (AROWS == 64)
        return bf ? kernel_ptr<128, true, 1, 64, false, true>() : kernel_ptr<128, false, 1, 64, false, true>();
    return bf ? kernel_ptr<128, true, 1, 128, false, true>() : kernel_ptr<128, false, 1, 128, false, true>();
}

template <int CM>
void* pick_kernel_cm(int BN, int dtype) {
    if (BN == 256)
        return dtype == GEMM_BF16 ? kernel_ptr<256, true, CM>() : kernel_ptr<256, false, CM>();
    return dtype == GEMM_BF16 ? kernel_ptr<128, true, CM>() : kernel_ptr<128, false, CM>();
}

void* pick_kernel(int BN, int dtype, int CM, int AROWS = 128, int PAIR = 0) {
    const bool bf = dtype == GEMM_BF16;
    if (PAIR) {  // CM = 2, BN = 128 or 256, AROWS = 128 or 64
        if (AROWS == 64) {
            if (BN == 256) return bf ? kernel_ptr<256, true, 2, 64, true>() : kernel_ptr<256, false, 2, 64, true>();
            return bf ? kernel_ptr<128, true, 2, 64, true>() : kernel_ptr<128, false, 2, 64, true>();
        }
        if (BN == 256) return bf ? kernel_ptr<256, true, 2, 128, true>() : kernel_ptr<256, false, 2, 128, true>();
        return bf ? kernel_ptr<128, true, 2, 128, true>() : kernel_ptr<128, false, 2, 128, true>();
    }
    if (BN == 64) {  // only with CM = 1
        if (AROWS == 64) return bf ? kernel_ptr<64, true, 1, 64>() : kernel_ptr<64, false, 1, 64>();
        return bf ? kernel_ptr<64, true, 1>() : kernel_ptr<64, false, 1>();
    }
    if (AROWS == 64) {  // BN = 128 or 256, CM = 1
        if (BN == 256) return bf ? kernel_ptr<256, true, 1, 64>() : kernel_ptr<256, false, 1, 64>();
        return bf ? kernel_ptr<128, true, 1, 64>() : kernel_ptr<128, false, 1, 64>();
    }
    return CM == 2 ? pick_kernel_cm<2>(BN, dtype) : pick_kernel_cm<1>(BN, dtype);
}

int kernel_index(int BN, int dtype, int CM, int AROWS, int PAIR, int KCL = 0) {
    const int bf = dtype == GEMM_BF16 ? 1 : 0;
    if (KCL) return 26 + 4 * (BN == 256 ? 1 : 0) + 2 * (AROWS == 64 ? 1 : 0) + bf;
    if (PAIR) return 14 + 4 * (AROWS == 64 ? 1 : 0) + 2 * (BN == 256 ? 1 : 0) + bf;
    if (BN == 64) return 10 + 2 * (AROWS == 64 ? 1 : 0) + bf;
    if (AROWS == 64) return (BN == 256 ? 22 : 8) + bf;
    return (BN == 256 ? 4 : 0) + 2 * bf + (CM == 2 ? 1 : 0);
}

int smem_for(int BN, int AROWS = 128, int PAIR = 0) {
    if (PAIR && AROWS == 64)
        return BN == 256 ? Cfg<256, 64, true>::SMEM_BYTES : Cfg<128, 64, true>::SMEM_BYTES;
    if (PAIR) return BN == 256 ? Cfg<256, 128, true>::SMEM_BYTES : Cfg<128, 128, true>::SMEM_BYTES;
    if (BN == 64) return AROWS == 64 ? Cfg<64, 64>::SMEM_BYTES : Cfg<64>::SMEM_BYTES;
    if (AROWS == 64) return BN == 256 ? Cfg<256, 64>::SMEM_BYTES : Cfg<128, 64>::SMEM_BYTES;
    return BN == 256 ? Cfg<256>::SMEM_BYTES : Cfg<128>::SMEM_BYTES;
}
int stages_for(int BN, int AROWS = 128, int PAIR = 0) {
    if (PAIR && AROWS == 64) return BN == 256 ? Cfg<256, 64, true>::STAGES : Cfg<128, 64, true>::STAGES;
    if (PAIR) return BN == 256 ? Cfg<256, 128, true>::STAGES : Cfg<128, 128, true>::STAGES;
    if (BN == 64) return AROWS == 64 ? Cfg<64, 64>::STAGES : Cfg<64>::STAGES;
    if (AROWS == 64) return BN == 256 ? Cfg<256, 64>::STAGES : Cfg<128, 64>::STAGES;
    return BN == 256 ? Cfg<256>::STAGES : Cfg<128>::STAGES;
}

// Clusters of S CTAs of the cluster split-K kernel (tile width BN, AROWS rows
// of A per stage) that can be resident at once on device `dev`: a cluster
// lives inside one GPC, so fewer than #SMs / S may fit.  0 when unknown.
int kcl_active_clusters(int dev, int BN, int dtype, int AROWS, int S) {
    static std::mutex mu;
    static int cache[64][2][2][3];  // device, BN == 256, AROWS == 64, S = 2 / 4 / 8
    if (dev < 0 || dev >= 64 || (S != 2 && S != 4 && S != 8)) return 0;
    const int si = S == 2 ? 0 : (S == 4 ? 1 : 2);
    std::lock_guard<std::mutex> lock(mu);
    int& c = cache[dev][BN == 256][AROWS == 64][si];
    if (c) return c;
    void* fn = pick_kernel_kcl(BN, dtype, AROWS);
    const int smem = smem_for(BN, AROWS, 0);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)S, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    c = n;
    return c;
}

// Cluster split-K: tile width and parts per tile.  Fixed options are kept
// (UNSUPPORTED when invalid); otherwise the pair with the most CTAs in one
// wave of g whose clusters can all be resident at once, preferring 256-wide
// tiles (512-byte runs of a row-major B), then more parts.  When no pair
// fits one wave: 256-wide tiles, 2 parts.
gemm_status_t kcl_shape(const gemm_plan* p, int64_t g, int* bn_out, int64_t* s_out,
                        bool* fits_out = nullptr) {
    const int64_t ipt = cdiv64(p->K, BK), tiles_m = cdiv64(p->M, BM);
    const int fixed_bn = p->opt_tile_n;
    const int64_t fixed_s = p->opt_split;
    if (fixed_bn == 64 || p->opt_cluster_m == 2) return GEMM_ERR_UNSUPPORTED;
    if (fixed_s != 0 && ((fixed_s != 2 && fixed_s != 4 && fixed_s != 8) || fixed_s > ipt))
        return GEMM_ERR_UNSUPPORTED;
    if (fixed_s == 0 && ipt < 2) return GEMM_ERR_UNSUPPORTED;
    const int bns[2] = {256, 128};
    const int64_t ss[3] = {8, 4, 2};
    int best_bn = fixed_bn ? fixed_bn : 256;
    int64_t best_s = fixed_s ? fixed_s : 2, best_ctas = -1;
    for (int bn : bns) {
        if (fixed_bn && bn != fixed_bn) continue;
        const int64_t tiles = tiles_m * cdiv64(p->N, bn);
        const int arows = (p->M <= 64) ? 64 : 128;
        for (int64_t S : ss) {
            if ((fixed_s && S != fixed_s) || S > ipt) continue;
            const int64_t ctas = tiles * S;
            if (ctas > g) continue;
            const int resident = p->offline ? (int)(p->num_sms / S)
                                            : kcl_active_clusters(p->device, bn, p->dtype, arows, (int)S);
            if (resident > 0 && tiles > resident) continue;
            if (ctas > best_ctas) {
                best_ctas = ctas;
                best_bn = bn;
                best_s = S;
            }
        }
    }
    *bn_out = best_bn;
    *s_out = best_s;
    if (fits_out) *fits_out = best_ctas > 0;
    return GEMM_OK;
}

// Derive the tile grid and the schedule from the shape and the options
// (issue "Stream-k matmul implementation very slow ...", final version,
// wrapper: tile counts, Stream-K tile count with the two_tiles rule, even
// split of the Stream-K iterations).
gemm_status_t derive(gemm_plan* p) {
    const int64_t tiles_m128 = cdiv64(p->M, BM);
    // cluster split-K: the k-parts of a tile run as one cluster of 1-CTA MMAs.
    // GEMM_SCHED_AUTO takes it when some choice of it fits one wave:
    //  * for a single row of 128-row tiles (a skinny, memory-bound product)
    //    when K has more than 16 k-blocks and the unsplit 128-wide tiles
    //    would fill under 80 % of the SMs.  In a timed sweep of 45 such
    //    shapes (M 16-128, N 1024-16384, K 1024-16384) it was never slower
    //    than Stream-K and up to 2.8x faster; with 16 k-blocks (K = 1024) the
    //    unsplit tiles ran 10-35 % faster, and with N = 16384 (128 tiles) they
    //    were level or up to 12 % faster;
    //  * for more rows when every part has at least 8 k-blocks: on the
    //    log-sampled shapes where it fits one wave it was 8-43 % faster than
    //    the other schedules with parts of 11-46 k-blocks, 25 % slower with 6.
    const int64_t g_kcl = p->opt_grid > 0 ? p->opt_grid : p->num_sms;
    bool kcl = p->schedule == GEMM_SCHED_SPLITK && p->opt_split_cluster == 1;
    int kcl_bn = 0;
    int64_t kcl_s = 0;
    if (kcl) {
        const gemm_status_t st = kcl_shape(p, g_kcl, &kcl_bn, &kcl_s);
        if (st != GEMM_OK) return st;
    } else if (p->schedule == GEMM_SCHED_AUTO && p->K > BK && p->opt_cluster_m != 2 &&
               p->opt_tile_n != 64) {
        bool fits = false;
        gemm_plan q = *p;
        q.opt_split = 0;  // the split-K part count does not apply to the other schedules
        const int64_t kblocks = cdiv64(p->K, BK);
        const bool single_row_ok = kblocks > 16 && cdiv64(p->N, 128) * 5 < 4 * g_kcl;
        if (kcl_shape(&q, g_kcl, &kcl_bn, &kcl_s, &fits) == GEMM_OK && fits &&
            (tiles_m128 == 1 ? single_row_ok : kblocks >= 8 * kcl_s))
            kcl = true;
    }
    // Tile width: 256 when that still gives every SM a tile (compute-bound
    // shapes: fewest operand bytes per FLOP); 64 for small problems with
    // several rows of tiles that would leave most SMs idle at 128 (more tiles
    // instead of a split of K); else 128.  A single row of tiles streams a B
    // that is read once and keeps 128: 256-byte runs per row of a row-major B
    // stream about twice as fast as 128-byte ones.
    int BN = kcl ? kcl_bn : p->opt_tile_n;
    if (BN == 0) {
        const int64_t tiles256 = tiles_m128 * cdiv64(p->N, 256);
        const int64_t tiles128 = tiles_m128 * cdiv64(p->N, 128);
        if (p->N > 128 && tiles256 >= p->num_sms) BN = 256;
        else if (p->N <= 64 || (tiles_m128 >= 2 && 2 * tiles128 < p->num_sms)) BN = 64;
        else BN = 128;
        if (BN == 64 && p->opt_cluster_m == 2) BN = 128;  // clusters need 128+ wide tiles
    }
    // 2-CTA clusters share B between two 128-row halves: worth it when there
    // are at least two row tiles and the tile is wide (compute-bound shapes)
    int CM = p->opt_cluster_m;
    if (CM == 0) CM = (tiles_m128 >= 2 && BN == 256 && !kcl) ? 2 : 1;
    if (BN == 64 && CM == 2) return GEMM_ERR_UNSUPPORTED;  // 64-wide tiles run without clusters
    // the scheduler works on tiles of CM*128 rows and on units of CM CTAs
    const int64_t tiles_m = cdiv64(p->M, (int64_t)BM * CM);
    const int64_t tiles_n = cdiv64(p->N, BN);
    const int64_t tiles = tiles_m * tiles_n;
    const int64_t ipt = cdiv64(p->K, BK);
    if (tiles > INT32_MAX / 2 || ipt > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;

    int g_ctas = p->opt_grid > 0 ? p->opt_grid : p->num_sms;
    if (CM == 2 && p->max_pair_ctas > 0 && g_ctas > p->max_pair_ctas) g_ctas = p->max_pair_ctas;
    const int g = g_ctas / CM > 0 ? g_ctas / CM : 1;  // scheduling units

    // GEMM_SCHED_AUTO: choose from the shape, after a timed sweep of 30
    // log-sampled shapes and the five workloads on GB300:
    //  * one row of tiles (skinny, memory-bound) under one wave -> Stream-K,
    //    whose units start at different k and so spread the B stream; but
    //    persistent (unsplit tiles) when K has at most 16 k-blocks or the
    //    tiles fill 80 % of the SMs (the timed sweep of single-row shapes:
    //    10-35 % and up to 12 % faster than Stream-K there);
    //  * fewer than 8 k-iterations per unit -> persistent (nothing to split);
    //  * four or more waves of tiles -> the hybrid rule, which removes the
    //    last partial wave, when tiles have at least 64 k-iterations or there
    //    are at least 12 waves; else persistent (few waves of short tiles put
    //    a large share of the work in short split units);
    //  * under one wave -> Stream-K when at most 70% of the units would have
    //    a tile, else persistent (the fixup costs more than the idle units);
    //  * one to four waves -> the hybrid rule when each split tile has at most
    //    8 contributors and tiles have at least 32 k-iterations (it keeps most
    //    tiles whole), else every tile in the Stream-K wave (a few tiles split
    //    many ways make their owners add a dozen partials).
    int sched = p->schedule;
    int sk_mode = p->opt_sk_mode;
    if (sched == GEMM_SCHED_AUTO && kcl) {
        sched = GEMM_SCHED_SPLITK;
    } else if (sched == GEMM_SCHED_AUTO) {
        const double waves = (double)tiles / g;
        int64_t sk_h = tiles % g;
        if (tiles - sk_h > g) sk_h += g;
        if (tiles_m == 1 && tiles < g) {
            sched = (ipt <= 16 || tiles * 5 >= 4 * (int64_t)g) ? GEMM_SCHED_PERSISTENT
                                                               : GEMM_SCHED_STREAMK;
        } else if (tiles * ipt < 8 * (int64_t)g) {
            sched = GEMM_SCHED_PERSISTENT;
        } else if (waves >= 4.0) {
            sched = (ipt >= 64 || waves >= 12.0) ? GEMM_SCHED_STREAMK : GEMM_SCHED_PERSISTENT;
            sk_mode = 0;
        } else if (waves < 1.0) {
            sched = (tiles * 10 <= 7 * (int64_t)g) ? GEMM_SCHED_STREAMK : GEMM_SCHED_PERSISTENT;
        } else {
            sched = GEMM_SCHED_STREAMK;
            const bool hybrid_ok = sk_h > 0 && g <= 8 * sk_h && ipt >= 32;
            sk_mode = hybrid_ok ? 0 : 1;
        }
    }
    p->eff_schedule = sched;
    p->eff_sk_mode = sk_mode;

    Sched s{};
    s.tiles_m = (int32_t)tiles_m;
    s.tiles_n = (int32_t)tiles_n;
    s.tiles = (int32_t)tiles;
    s.ipt = (int32_t)(ipt > 0 ? ipt : 1);
    s.group_m = p->opt_group_m >= 0 ? p->opt_group_m
                                    : (sched == GEMM_SCHED_DATA_PARALLEL ? 0 : 8);
    s.sk_tiles = 0;
    s.sk_q = s.sk_r = 0;
    if (sched == GEMM_SCHED_DATA_PARALLEL) {
        s.grid = s.tiles;
        s.persistent = 0;
    } else if (sched == GEMM_SCHED_PERSISTENT) {
        s.grid = (int32_t)(tiles < g ? tiles : g);
        s.persistent = 1;
    } else if (sched == GEMM_SCHED_SPLITK && kcl) {
        // S parts per tile, each a CTA of the tile's cluster (kcl_shape)
        const int64_t S = kcl_s;
        if (tiles * S > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;
        s.kc = (int32_t)S;
        s.grid = (int32_t)(tiles * S);
        s.persistent = 0;
    } else if (sched == GEMM_SCHED_SPLITK) {
        // as many parts as fit in one round of the scheduling units, at most
        // one part per 4 k-iterations
        int64_t S = p->opt_split;
        if (S == 0) {
            S = tiles >= g ? 1 : g / tiles;
            const int64_t cap = ipt / 4 > 1 ? ipt / 4 : 1;
            if (S > cap) S = cap;
        }
        if (S > ipt) S = ipt > 0 ? ipt : 1;
        if (tiles * S > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;
        s.split = (int32_t)S;
        s.grid = (int32_t)(tiles * S < g ? tiles * S : g);
        s.persistent = 1;
    } else {
        int64_t sk = tiles % g;
        if (p->opt_two_tiles && tiles - sk > g) sk += g;
        if (sk_mode == 1) sk = tiles;  // every tile in the Stream-K wave
        s.sk_tiles = (int32_t)sk;
        s.grid = tiles > 0 ? g : 0;
        s.persistent = 1;
        const int64_t iters = sk * (int64_t)s.ipt;
        s.sk_q = iters / g;
        s.sk_r = iters % g;
    }
    s.k_rotate = p->opt_k_rotate > 0 ? 1 : 0;
    s.raster_table = nullptr;  // the device / host tables are set where the Sched is used
    if (p->opt_raster == 1) {
        if (tiles_m > 65535 || tiles_n > 65535) return GEMM_ERR_UNSUPPORTED;
        if (!p->raster_host) p->raster_host = new (std::nothrow) std::vector<int32_t>();
        if (!p->raster_host) return GEMM_ERR_CUDA;
        hilbert_order(tiles_m, tiles_n, *p->raster_host);
        if (!p->offline) {
            // uploaded here, at configuration time, so that running allocates nothing
            if (p->raster_dev && p->raster_tiles < tiles) {
                cudaFree(p->raster_dev);
                p->raster_dev = nullptr;
            }
            if (!p->raster_dev && tiles > 0) {
                if (cudaMalloc(&p->raster_dev, (size_t)tiles * sizeof(int32_t)) != cudaSuccess) {
                    p->raster_dev = nullptr;
                    return GEMM_ERR_CUDA;
                }
                p->raster_tiles = tiles;
            }
            if (tiles > 0 && cudaMemcpy(p->raster_dev, p->raster_host->data(),
                                        (size_t)tiles * sizeof(int32_t),
                                        cudaMemcpyHostToDevice) != cudaSuccess)
                return GEMM_ERR_CUDA;
        }
    }
    // off by default: measured slower on a B read once (extra L2 requests)
    s.l2_prefetch = p->opt_l2_prefetch > 0 ? p->opt_l2_prefetch : 0;
    p->s = s;
    p->BN = BN;
    p->CM = CM;
    // one row of tiles with at most 64 valid rows: load only those rows of A
    // pair MMA (tcgen05 cta_group::2) for 2-CTA clusters: each CTA keeps
    // only its half of B, so the ring is deeper
    p->PAIR = (CM == 2 && p->opt_pair_mma == 1) ? 1 : 0;
    // at most 64 valid rows: load only 64 rows of A per stage (without
    // clusters, or with a pair MMA)
    p->AROWS = (p->M <= 64 && (CM == 1 || p->PAIR)) ? 64 : 128;
    p->ctas = s.grid * CM;
    p->stages = stages_for(BN, p->AROWS, p->PAIR);
    p->smem_bytes = smem_for(BN, p->AROWS, p->PAIR);
    if (sched == GEMM_SCHED_STREAMK && s.sk_tiles > 0) {
        // the hybrid rule splits fewer than 2g tiles whatever the shape: size
        // the flags for 2g, so a plan over a block of this product (same grid)
        // fits this workspace
        const int64_t flag_tiles = sk_mode == 1 ? s.sk_tiles : std::max<int64_t>(s.sk_tiles, 2 * (int64_t)g);
        p->ws_flag_bytes = ((size_t)flag_tiles * CM * 8 + 255) / 256 * 256;
        p->ws_bytes = p->ws_flag_bytes + (size_t)p->ctas * BM * BN * sizeof(float);
    } else if (sched == GEMM_SCHED_SPLITK && s.split > 1) {
        // one flag per tile half, one partial slot per (tile, part >= 1, half)
        p->ws_flag_bytes = ((size_t)s.tiles * CM * 8 + 255) / 256 * 256;
        p->ws_bytes = p->ws_flag_bytes +
                      (size_t)s.tiles * (s.split - 1) * CM * BM * BN * sizeof(float);
    } else {
        p->ws_flag_bytes = 0;
        p->ws_bytes = 0;
    }
    p->tm_valid = false;
    p->tm_c_state = 0;
    return GEMM_OK;
}

// k-blocks of each CTA's first unit prefetched into L2 before the wait for the
// previous kernel.  Default: 8 when the launch fills at least three quarters
// of the SMs, else none.  Paired bursts on GB300 with 8: 2.8 % faster on
// 2304 x 2304 x 8192 (all-tiles Stream-K), 3.6-4.6 % on two log-sampled
// shapes, 1.6 % on the skinny cluster split-K, within noise on 8192^3; but
// 9.7 % slower on a 64-CTA launch (16 x 1024 x 4096), whose successor's CTAs
// all start early on idle SMs and prefetch while it still streams.  16 or
// more k-blocks were slower on the skinny product (the prefetch crowds L2).
int early_prefetch_of(const gemm_plan* p) {
    if (p->opt_early_prefetch >= 0) return p->opt_early_prefetch;
    return 4 * (int64_t)p->ctas >= 3 * (int64_t)p->num_sms ? 8 : 0;
}

// CTAs that can be resident at once as 2-CTA clusters of the (largest) kernel
// configuration; clusters live inside one GPC, so this can be below #SMs.
int max_pair_ctas(int dev) {
    static std::mutex mu;
    static int cache[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev]) return cache[dev];
    void* fn = pick_kernel(256, GEMM_BF16, 2);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_for(256)) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem_for(256);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cache[dev] = 2 * n;
    return cache[dev];
}

gemm_status_t make_plan(gemm_plan_t* out, int64_t M, int64_t N, int64_t K, int dtype, int la,
                        int lb, int sched, int offline, int num_sms) {
    if (!out || M < 0 || N < 0 || K < 0 || !valid_enums(dtype, la, lb, sched))
        return GEMM_ERR_INVALID_ARG;
    gemm_plan* p = new (std::nothrow) gemm_plan();
    if (!p) return GEMM_ERR_CUDA;
    p->M = M;
    p->N = N;
    p->K = K;
    p->dtype = dtype;
    p->layout_a = la;
    p->layout_b = lb;
    p->schedule = sched;
    p->offline = offline;
    p->opt_grid = 0;
    p->opt_group_m = -1;
    p->opt_tile_n = 0;
    p->opt_two_tiles = 1;
    p->inject_skip = -1;
    p->opt_cluster_m = 0;
    p->opt_sk_mode = 0;
    p->opt_split = 0;
    p->opt_k_rotate = 0;
    p->opt_l2_prefetch = -1;
    p->opt_pair_mma = 1;
    p->opt_early_prefetch = -1;
    p->opt_split_cluster = 0;
    p->opt_raster = 0;
    p->wait_limit_us = 1000000;
    p->a_ld = 0;
    p->opt_host_chunks = 0;
    p->opt_host_col_chunks = 0;
    p->owns_status = true;
    if (offline) {
        if (num_sms <= 0) { delete p; return GEMM_ERR_INVALID_ARG; }
        p->device = -1;
        p->num_sms = num_sms;
    } else {
        int dev = 0, count = 0;
        if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
            cudaGetLastError();
            delete p;
            return GEMM_ERR_NO_DEVICE;
        }
        int major = 0, minor = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            delete p;
            return GEMM_ERR_CUDA;
        }
        if (major != 10 || minor != 3) { delete p; return GEMM_ERR_NO_DEVICE; }
        p->device = dev;
        p->num_sms = sms;
        p->max_pair_ctas = max_pair_ctas(dev);
        if (cudaMalloc(&p->d_status, sizeof(int)) != cudaSuccess ||
            cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) {
            if (p->d_status) cudaFree(p->d_status);
            delete p;
            return GEMM_ERR_CUDA;
        }
    }
    gemm_status_t st = derive(p);
    if (st != GEMM_OK) {
        if (p->d_status) cudaFree(p->d_status);
        delete p;
        return st;
    }
    if (getenv("GEMM_DEBUG")) {
        fprintf(stderr,
                "[gemm] M=%lld N=%lld K=%lld dtype=%d A=%s B=%s sched=%d | tile %dx%dx64 "
                "(cluster %d) tiles %dx%d=%d ipt=%d units=%d ctas=%d sk_tiles=%d sk_q=%lld "
                "sk_r=%lld group_m=%d ws=%zu smem=%d pair_ctas=%d\n",
                (long long)M, (long long)N, (long long)K, dtype, la ? "col" : "row",
                lb ? "col" : "row", sched, BM * p->CM, p->BN, p->CM, p->s.tiles_m, p->s.tiles_n,
                p->s.tiles, p->s.ipt, p->s.grid, p->ctas, p->s.sk_tiles, (long long)p->s.sk_q,
                (long long)p->s.sk_r, p->s.group_m, p->ws_bytes, p->smem_bytes, p->max_pair_ctas);
    }
    *out = p;
    return GEMM_OK;
}

// Tensor map of C for the whole-tile stores of the pair-MMA kernels:
// row-major, dims {N, M}, row stride ldc, boxes of 64 columns x 32 rows with
// the 128-byte swizzle (the epilogue stages each box in that layout).  It
// needs a 16-byte aligned C and a row stride that is a multiple of 16 bytes;
// otherwise (and for the other kernels) C is written with vector stores.
bool encode_c_map(gemm_plan* p, void* C, int64_t ldc) {
    if (!p->PAIR || !C) return false;
    if (p->tm_c_state != 0 && p->tm_c_ptr == C && p->tm_c_ld == ldc) return p->tm_c_state > 0;
    p->tm_c_ptr = C;
    p->tm_c_ld = ldc;
    p->tm_c_state = -1;
    if (((uintptr_t)C & 15u) || ((ldc * 2) & 15)) return false;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const CUtensorMapDataType dt =
        p->dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[2] = {(cuuint64_t)p->N, (cuuint64_t)p->M};
    const cuuint64_t strides[1] = {(cuuint64_t)ldc * 2};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&p->tmC, dt, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    p->tm_c_state = 1;
    return true;
}

gemm_status_t encode_maps(gemm_plan* p, const void* A, const void* B) {
    if (p->tm_valid && p->tm_a_ptr == A && p->tm_b_ptr == B) return GEMM_OK;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return GEMM_ERR_CUDA;
    const CUtensorMapDataType dt =
        p->dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint32_t estr[2] = {1, 1};
    // A: row-major M x K -> dims {K, M}, box {64, 128}; column-major -> dims {M, K}, box {64, 64}
    {
        cuuint64_t dims[2], strides[1];
        cuuint32_t box[2];
        if (p->layout_a == GEMM_ROW_MAJOR) {
            dims[0] = (cuuint64_t)p->K; dims[1] = (cuuint64_t)p->M;
            strides[0] = (cuuint64_t)p->K * 2;
            box[0] = BK; box[1] = (cuuint32_t)p->AROWS;
        } else {
            dims[0] = (cuuint64_t)p->M; dims[1] = (cuuint64_t)p->K;
            strides[0] = (cuuint64_t)(p->a_ld ? p->a_ld : p->M) * 2;
            box[0] = 64; box[1] = BK;
        }
        if (enc(&p->tmA, dt, 2, const_cast<void*>(A), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GEMM_ERR_UNSUPPORTED;
    }
    // B: column-major K x N (stored N x K) -> dims {K, N}, box {64, BN};
    //    row-major K x N -> dims {N, K}, box {64, 64}
    {
        cuuint64_t dims[2], strides[1];
        cuuint32_t box[2];
        if (p->layout_b == GEMM_COL_MAJOR) {
            dims[0] = (cuuint64_t)p->K; dims[1] = (cuuint64_t)p->N;
            strides[0] = (cuuint64_t)p->K * 2;
            box[0] = BK; box[1] = (cuuint32_t)(p->BN / p->CM);  // each CTA of a pair loads half
        } else {
            dims[0] = (cuuint64_t)p->N; dims[1] = (cuuint64_t)p->K;
            strides[0] = (cuuint64_t)(p->b_ld ? p->b_ld : p->N) * 2;
            box[0] = 64; box[1] = BK;
        }
        if (enc(&p->tmB, dt, 2, const_cast<void*>(B), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GEMM_ERR_UNSUPPORTED;
    }
    p->tm_a_ptr = A;
    p->tm_b_ptr = B;
    p->tm_valid = true;
    return GEMM_OK;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

gemm_status_t run_impl(gemm_plan_t p, const void* A, const void* B, void* C, void* workspace,
                       gemm_stream_t stream, bool pdl);

// Options of a sub-plan over a block of the parent's product: the same tile
// shape, cluster, schedule and options; A, B and C keep the parent's leading
// dimensions.
void sub_options(const gemm_plan* p, gemm_plan* sp) {
    sp->opt_grid = p->opt_grid;
    sp->opt_group_m = p->opt_group_m;
    sp->opt_tile_n = p->BN;
    sp->opt_two_tiles = p->opt_two_tiles;
    sp->opt_cluster_m = p->CM;
    sp->opt_sk_mode = p->eff_sk_mode;
    // split-K: the parent's resolved part count, so every block sums in the
    // parent's order (and a parent without partials gets sub-plans without)
    sp->opt_split = p->eff_schedule == GEMM_SCHED_SPLITK ? p->s.split : p->opt_split;
    sp->opt_k_rotate = p->opt_k_rotate;
    sp->opt_l2_prefetch = p->opt_l2_prefetch;
    sp->opt_pair_mma = p->opt_pair_mma;
    sp->opt_split_cluster = p->s.kc > 0 ? 1 : p->opt_split_cluster;  // AUTO may have chosen it
    sp->opt_early_prefetch = p->opt_early_prefetch;
    if (p->s.kc > 0) sp->opt_split = p->s.kc;
    sp->wait_limit_us = p->wait_limit_us;
    sp->a_ld = p->layout_a == GEMM_COL_MAJOR ? (p->a_ld ? p->a_ld : p->M) : 0;
    sp->b_ld = p->layout_b == GEMM_ROW_MAJOR ? (p->b_ld ? p->b_ld : p->N) : 0;
    sp->c_ld = p->c_ld ? p->c_ld : p->N;
}

// Workspace of a sub-plan over a rows x cols block, from a scratch copy of
// the plan (no raster table: it does not change the sizes and the copy builds
// none).
bool sub_workspace(const gemm_plan* p, int64_t rows, int64_t cols, size_t* flag_bytes,
                   size_t* part_bytes) {
    gemm_plan tmp = *p;
    tmp.raster_host = nullptr;
    tmp.raster_dev = nullptr;
    tmp.opt_raster = 0;
    tmp.M = rows;
    tmp.N = cols;
    tmp.schedule = p->eff_schedule;
    sub_options(p, &tmp);
    if (derive(&tmp) != GEMM_OK) return false;
    *flag_bytes = tmp.ws_flag_bytes;
    *part_bytes = tmp.ws_bytes - tmp.ws_flag_bytes;
    return true;
}

// gemm_run_host: the block grid.  Row chunks are whole scheduled tile rows,
// column chunks whole tile columns.  By default: with M >= 2048, row chunks
// (at least 512 rows each, at most 8), which start after B has arrived; when
// B is the larger operand (N > M), blocks of about a quarter of each side
// instead, which start once one chunk of A and one of B have arrived; with
// only N >= 2048, column chunks; serial otherwise.  The
// sub-plans must fit the plan's workspace: their partials after one flag
// region as large as any of them needs.
int host_grid(const gemm_plan* p, int64_t* rows_out, int64_t* cols_out, int* nr_out, int* nc_out) {
    int nr = 1, nc = 1;
    if (p->M > 0 && p->N > 0 && p->K > 0) {
        // a row chunk needs all of B and a column chunk all of A before its
        // first block: split both sides only when B is the larger operand
        const bool two_d = p->M >= 2048 && p->N > p->M;
        if (p->opt_host_chunks >= 2)
            nr = p->opt_host_chunks;
        else if (p->opt_host_chunks == 0 && p->M >= 2048)
            nr = (int)std::min<int64_t>(two_d ? 4 : 8, p->M / (two_d ? 1024 : 512));
        if (p->opt_host_col_chunks >= 2)
            nc = p->opt_host_col_chunks;
        else if (p->opt_host_col_chunks == 0 && p->N >= 2048 && (two_d || p->M < 2048))
            nc = (int)std::min<int64_t>(two_d ? 4 : 8, p->N / (two_d ? 1024 : 512));
    }
    const int64_t unit_m = (int64_t)BM * p->CM, unit_n = p->BN > 0 ? p->BN : 128;
    int64_t rows = p->M, cols = p->N;
    if (nr > 1) {
        rows = ((p->M + nr - 1) / nr + unit_m - 1) / unit_m * unit_m;
        nr = (int)((p->M + rows - 1) / rows);
    }
    if (nc > 1) {
        cols = ((p->N + nc - 1) / nc + unit_n - 1) / unit_n * unit_n;
        nc = (int)((p->N + cols - 1) / cols);
    }
    if (nr < 1) nr = 1;
    if (nc < 1) nc = 1;
    if (nr == 1) rows = p->M;
    if (nc == 1) cols = p->N;
    while (nr * nc > 64) {  // events for at most 64 blocks
        if (nc > 1) {
            cols *= 2;
            nc = (int)((p->N + cols - 1) / cols);
        } else {
            rows *= 2;
            nr = (int)((p->M + rows - 1) / rows);
        }
    }
    if (nr * nc > 1) {
        size_t f = 0, q = 0;
        const int64_t rs[2] = {rows, p->M % rows}, cs[2] = {cols, p->N % cols};
        for (int i = 0; i < 2 && nr * nc > 1; ++i)
            for (int j = 0; j < 2 && nr * nc > 1; ++j) {
                if (rs[i] == 0 || cs[j] == 0) continue;
                size_t fb = 0, pb = 0;
                if (!sub_workspace(p, rs[i], cs[j], &fb, &pb)) {
                    nr = nc = 1;
                    break;
                }
                f = std::max(f, fb);
                q = std::max(q, pb);
            }
        if (f + q > p->ws_bytes) nr = nc = 1;
    }
    if (nr * nc <= 1) {
        nr = nc = 1;
        rows = p->M;
        cols = p->N;
    }
    if (rows_out) *rows_out = rows;
    if (cols_out) *cols_out = cols;
    if (nr_out) *nr_out = nr;
    if (nc_out) *nc_out = nc;
    return nr * nc;
}

// A sub-plan over a rows x cols block; device errors land in the parent's
// status word.
gemm_status_t make_sub(gemm_plan* p, int64_t rows, int64_t cols, gemm_plan** out) {
    gemm_plan* sp = nullptr;
    gemm_status_t st = make_plan(&sp, rows, cols, p->K, p->dtype, p->layout_a, p->layout_b,
                                 p->eff_schedule, 0, 0);
    if (st != GEMM_OK) return st;
    sub_options(p, sp);
    sp->opt_raster = p->opt_raster;
    st = derive(sp);
    if (st != GEMM_OK) {
        gemm_plan_destroy(sp);
        return st;
    }
    cudaFree(sp->d_status);
    sp->d_status = p->d_status;
    sp->owns_status = false;
    *out = sp;
    return GEMM_OK;
}

void pipe_release(gemm_plan* p) {
    for (gemm_plan*& sp : p->sub) {
        if (sp) gemm_plan_destroy(sp);
        sp = nullptr;
    }
    // every handle is null until created, so a partly made pipeline is freed too
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    if (p->ev_start) cudaEventDestroy(p->ev_start);
    if (p->ev_done) cudaEventDestroy(p->ev_done);
    for (cudaEvent_t& e : p->ev_a) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
    }
    for (cudaEvent_t& e : p->ev_b) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
    }
    for (cudaEvent_t& e : p->ev_c) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
    }
    p->h2d = p->d2h = nullptr;
    p->ev_start = p->ev_done = nullptr;
    p->pipe_ready = false;
    p->sub_rows = p->sub_cols = 0;
}

gemm_status_t pipe_prepare(gemm_plan* p, int64_t rows, int64_t cols) {
    if (p->pipe_ready && p->sub_rows == rows && p->sub_cols == cols) return GEMM_OK;
    pipe_release(p);
    const unsigned ev_flags = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&p->ev_start, ev_flags) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&p->ev_done, ev_flags) == cudaSuccess;
    for (cudaEvent_t& e : p->ev_a) ok = ok && cudaEventCreateWithFlags(&e, ev_flags) == cudaSuccess;
    for (cudaEvent_t& e : p->ev_b) ok = ok && cudaEventCreateWithFlags(&e, ev_flags) == cudaSuccess;
    for (cudaEvent_t& e : p->ev_c) ok = ok && cudaEventCreateWithFlags(&e, ev_flags) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        pipe_release(p);
        return GEMM_ERR_CUDA;
    }
    p->pipe_ready = true;
    p->sub_rows = rows;
    p->sub_cols = cols;
    const int64_t rs[2] = {rows, p->M % rows}, cs[2] = {cols, p->N % cols};
    gemm_status_t st = GEMM_OK;
    for (int i = 0; i < 2 && st == GEMM_OK; ++i)
        for (int j = 0; j < 2 && st == GEMM_OK; ++j)
            if (rs[i] > 0 && cs[j] > 0 && !(rows == p->M && i == 1) && !(cols == p->N && j == 1))
                st = make_sub(p, rs[i], cs[j], &p->sub[2 * i + j]);
    if (st != GEMM_OK) {
        pipe_release(p);
        return st;
    }
    // the sub-plans share the caller's workspace: one flag region, as large
    // as any of them needs, then the partials (host_grid checked that it fits)
    size_t flags = 0;
    for (gemm_plan* sp : p->sub)
        if (sp) flags = std::max(flags, sp->ws_flag_bytes);
    for (gemm_plan* sp : p->sub)
        if (sp && sp->ws_bytes > 0) {
            sp->ws_bytes = flags + (sp->ws_bytes - sp->ws_flag_bytes);
            sp->ws_flag_bytes = flags;
        }
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_status_t gemm_plan_create(gemm_plan_t* out, int64_t M, int64_t N, int64_t K,
                               gemm_dtype_t dtype, gemm_layout_t layout_a, gemm_layout_t layout_b,
                               gemm_schedule_t schedule) {
    return make_plan(out, M, N, K, dtype, layout_a, layout_b, schedule, 0, 0);
}

gemm_status_t gemm_plan_create_offline(gemm_plan_t* out, int64_t M, int64_t N, int64_t K,
                                       gemm_dtype_t dtype, gemm_layout_t layout_a,
                                       gemm_layout_t layout_b, gemm_schedule_t schedule,
                                       int num_sms) {
    return make_plan(out, M, N, K, dtype, layout_a, layout_b, schedule, 1, num_sms);
}

gemm_status_t gemm_plan_set_option(gemm_plan_t p, int key, int64_t value) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    gemm_plan saved = *p;
    switch (key) {
        case GEMM_OPT_GRID:
            if (value < 0 || value > 65535) return GEMM_ERR_UNSUPPORTED;
            if ((p->schedule == GEMM_SCHED_STREAMK || p->schedule == GEMM_SCHED_AUTO) &&
                value > p->num_sms)
                return GEMM_ERR_UNSUPPORTED;
            p->opt_grid = (int)value;
            break;
        case GEMM_OPT_GROUP_M:
            if (value < 0 || value > 4096) return GEMM_ERR_UNSUPPORTED;
            p->opt_group_m = (int)value;
            break;
        case GEMM_OPT_TILE_N:
            if (value != 0 && value != 64 && value != 128 && value != 256) return GEMM_ERR_UNSUPPORTED;
            p->opt_tile_n = (int)value;
            break;
        case GEMM_OPT_TWO_TILES:
            if (value != 0 && value != 1) return GEMM_ERR_UNSUPPORTED;
            p->opt_two_tiles = (int)value;
            break;
        case GEMM_OPT_WAIT_LIMIT_US:
            if (value < 1 || value > 60000000) return GEMM_ERR_UNSUPPORTED;
            p->wait_limit_us = value;
            return GEMM_OK;
        case GEMM_OPT_INJECT_SKIP_POST:
            if (value < -1 || value > 65535) return GEMM_ERR_UNSUPPORTED;
            p->inject_skip = (int)value;
            return GEMM_OK;
        case GEMM_OPT_CLUSTER_M:
            if (value != 0 && value != 1 && value != 2) return GEMM_ERR_UNSUPPORTED;
            p->opt_cluster_m = (int)value;
            break;
        case GEMM_OPT_SK_MODE:
            if (value != 0 && value != 1) return GEMM_ERR_UNSUPPORTED;
            p->opt_sk_mode = (int)value;
            break;
        case GEMM_OPT_SPLIT_K:
            if (value < 0 || value > 4096) return GEMM_ERR_UNSUPPORTED;
            p->opt_split = (int)value;
            break;
        case GEMM_OPT_K_ROTATE:
            if (value < 0 || value > 1) return GEMM_ERR_UNSUPPORTED;
            p->opt_k_rotate = (int)value;
            break;
        case GEMM_OPT_L2_PREFETCH:
            if (value < 0 || value > 256) return GEMM_ERR_UNSUPPORTED;
            p->opt_l2_prefetch = (int)value;
            break;
        case GEMM_OPT_PAIR_MMA:
            if (value != 0 && value != 1) return GEMM_ERR_UNSUPPORTED;
            p->opt_pair_mma = (int)value;
            break;
        case GEMM_OPT_RASTER:
            if (value != 0 && value != 1) return GEMM_ERR_UNSUPPORTED;
            p->opt_raster = (int)value;
            break;
        case GEMM_OPT_HOST_CHUNKS:
            if (value < 0 || value > 16) return GEMM_ERR_UNSUPPORTED;
            p->opt_host_chunks = (int)value;
            break;
        case GEMM_OPT_HOST_COL_CHUNKS:
            if (value < 0 || value > 16) return GEMM_ERR_UNSUPPORTED;
            p->opt_host_col_chunks = (int)value;
            break;
        case GEMM_OPT_SPLIT_K_CLUSTER:
            if (value != 0 && value != 1) return GEMM_ERR_UNSUPPORTED;
            p->opt_split_cluster = (int)value;
            break;
        case GEMM_OPT_EARLY_PREFETCH:
            if (value < -1 || value > 256) return GEMM_ERR_UNSUPPORTED;
            p->opt_early_prefetch = (int)value;
            return GEMM_OK;
        default:
            return GEMM_ERR_INVALID_ARG;
    }
    gemm_status_t st = derive(p);
    if (st != GEMM_OK) {
        // the raster tables are reallocated in place: keep the current ones
        std::vector<int32_t>* rh = p->raster_host;
        int32_t* rd = p->raster_dev;
        int64_t rt = p->raster_tiles;
        *p = saved;
        p->raster_host = rh;
        p->raster_dev = rd;
        p->raster_tiles = rt;
        derive(p);  // the saved options derived before; rebuild any table for them
    } else {
        pipe_release(p);  // sub-plans follow the options: rebuilt on next use
    }
    return st;
}

gemm_status_t gemm_plan_get_info(gemm_plan_t p, int key, int64_t* value) {
    if (!p || !value) return GEMM_ERR_INVALID_ARG;
    int64_t v;
    switch (key) {
        case GEMM_INFO_TILE_M: v = (int64_t)BM * p->CM; break;
        case GEMM_INFO_TILE_N: v = p->BN; break;
        case GEMM_INFO_TILE_K: v = BK; break;
        case GEMM_INFO_TILES_M: v = p->s.tiles_m; break;
        case GEMM_INFO_TILES_N: v = p->s.tiles_n; break;
        case GEMM_INFO_TILES: v = p->s.tiles; break;
        case GEMM_INFO_ITERS_PER_TILE: v = cdiv64(p->K, BK); break;
        case GEMM_INFO_GRID: v = p->ctas; break;
        case GEMM_INFO_SK_TILES: v = p->s.sk_tiles; break;
        case GEMM_INFO_SK_ITERS_PER_CTA: v = p->s.sk_q; break;
        case GEMM_INFO_SK_ITERS_REM: v = p->s.sk_r; break;
        case GEMM_INFO_NUM_SMS: v = p->num_sms; break;
        case GEMM_INFO_STAGES: v = p->stages; break;
        case GEMM_INFO_GROUP_M: v = p->s.group_m; break;
        case GEMM_INFO_SMEM_BYTES: v = p->smem_bytes; break;
        case GEMM_INFO_CLUSTER_M: v = p->CM; break;
        case GEMM_INFO_A_ROWS_PER_STAGE: v = p->AROWS; break;
        case GEMM_INFO_SPLIT_K: v = p->s.kc > 0 ? p->s.kc : p->s.split; break;
        case GEMM_INFO_SPLIT_K_CLUSTER: v = p->s.kc > 0 ? 1 : 0; break;
        case GEMM_INFO_EARLY_PREFETCH: v = early_prefetch_of(p); break;
        case GEMM_INFO_CLUSTERS_RESIDENT:
            v = p->offline ? 0
                : p->s.kc > 0 ? kcl_active_clusters(p->device, p->BN, p->dtype, p->AROWS, p->s.kc)
                : p->CM == 2 ? max_pair_ctas(p->device) / 2 : 0;
            break;
        case GEMM_INFO_K_ROTATE: v = p->s.k_rotate; break;
        case GEMM_INFO_L2_PREFETCH: v = p->s.l2_prefetch; break;
        case GEMM_INFO_PAIR_MMA: v = p->PAIR; break;
        case GEMM_INFO_SCHEDULE: v = p->eff_schedule; break;
        case GEMM_INFO_RASTER: v = p->opt_raster; break;
        case GEMM_INFO_HOST_CHUNKS: {
            int nr = 1;
            host_grid(p, nullptr, nullptr, &nr, nullptr);
            v = nr;
            break;
        }
        case GEMM_INFO_HOST_COL_CHUNKS: {
            int nc = 1;
            host_grid(p, nullptr, nullptr, nullptr, &nc);
            v = nc;
            break;
        }
        case GEMM_INFO_SK_MODE: v = (p->eff_schedule == GEMM_SCHED_STREAMK && p->s.sk_tiles == p->s.tiles) ? 1 : 0; break;
        default: return GEMM_ERR_INVALID_ARG;
    }
    *value = v;
    return GEMM_OK;
}

gemm_status_t gemm_workspace_size(gemm_plan_t p, size_t* bytes) {
    if (!p || !bytes) return GEMM_ERR_INVALID_ARG;
    *bytes = p->ws_bytes;
    return GEMM_OK;
}

gemm_status_t gemm_run(gemm_plan_t p, const void* A, const void* B, void* C, void* workspace,
                       gemm_stream_t stream) {
    return run_impl(p, A, B, C, workspace, stream, true);
}

}  // extern "C"

namespace {

gemm_status_t run_impl(gemm_plan_t p, const void* A, const void* B, void* C, void* workspace,
                       gemm_stream_t stream, bool pdl) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (p->offline) return GEMM_ERR_NO_DEVICE;
    if (p->M == 0 || p->N == 0) return GEMM_OK;
    if (!C) return GEMM_ERR_INVALID_ARG;
    if (((uintptr_t)C & 15u) || (p->N % 8)) return GEMM_ERR_UNSUPPORTED;
    DeviceGuard guard(p->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (p->K == 0) {  // empty sum: C = +0
        const size_t ldc = (size_t)(p->c_ld ? p->c_ld : p->N);
        return cudaMemset2DAsync(C, ldc * 2, 0, (size_t)p->N * 2, (size_t)p->M, st) == cudaSuccess
                   ? GEMM_OK
                   : GEMM_ERR_CUDA;
    }
    if (!A || !B) return GEMM_ERR_INVALID_ARG;
    if (((uintptr_t)A & 15u) || ((uintptr_t)B & 15u) || (p->K % 8) ||
        (p->layout_a == GEMM_COL_MAJOR && ((p->a_ld ? p->a_ld : p->M) % 8)))
        return GEMM_ERR_UNSUPPORTED;
    if (p->ws_bytes > 0 && (!workspace || ((uintptr_t)workspace & 15u))) return GEMM_ERR_WORKSPACE;

    gemm_status_t es = encode_maps(p, A, B);
    if (es != GEMM_OK) return es;

    const int kcl = p->s.kc > 0 ? 1 : 0;
    void* fn = kcl ? pick_kernel_kcl(p->BN, p->dtype, p->AROWS)
                   : pick_kernel(p->BN, p->dtype, p->CM, p->AROWS, p->PAIR);
    const int bi = kernel_index(p->BN, p->dtype, p->CM, p->AROWS, p->PAIR, kcl);
    if (!p->attr_set[bi]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, p->smem_bytes) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
        p->attr_set[bi] = true;
    }
    if (p->ws_bytes > 0 && p->flags_cleared_for != workspace) {
        if (cudaMemsetAsync(workspace, 0, p->ws_flag_bytes, st) != cudaSuccess) return GEMM_ERR_CUDA;
        p->flags_cleared_for = workspace;
    }

    KParams kp{};
    kp.s = p->s;
    kp.s.raster_table = p->opt_raster == 1 ? p->raster_dev : nullptr;
    kp.M = (int32_t)p->M;
    kp.N = (int32_t)p->N;
    kp.K = (int32_t)p->K;
    kp.ldc = (int32_t)(p->c_ld ? p->c_ld : p->N);
    kp.C = C;
    kp.flags = p->ws_bytes ? reinterpret_cast<unsigned long long*>(workspace) : nullptr;
    kp.partials = p->ws_bytes
                      ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + p->ws_flag_bytes)
                      : nullptr;
    kp.status = p->d_status;
    kp.idesc = idesc_f16(p->dtype == GEMM_BF16, p->layout_a == GEMM_COL_MAJOR,
                         p->layout_b == GEMM_ROW_MAJOR, p->PAIR ? 2 * BM : BM, p->BN);
    kp.epoch = next_epoch();
    kp.a_mn = p->layout_a == GEMM_COL_MAJOR;
    kp.b_mn = p->layout_b == GEMM_ROW_MAJOR;
    kp.inject_skip_cta = p->inject_skip;
    kp.wait_limit_ns = (uint64_t)p->wait_limit_us * 1000ull;
    kp.pipe_limit_ns = 4000000000ull;
    kp.trace = (p->trace && p->trace_bytes >= (size_t)p->ctas * TRACE_N * 8) ? p->trace : nullptr;
    kp.early_prefetch = early_prefetch_of(p);
    kp.c_tma = encode_c_map(p, C, kp.ldc) ? 1 : 0;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p->ctas, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)p->smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (p->CM == 2 || kcl) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = kcl ? (unsigned)p->s.kc : 2u;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    // Programmatic dependent launch: this grid may start while the previous
    // kernel in the stream drains; the kernel waits (griddepcontrol.wait)
    // before touching global memory.  Off for the host pipeline's chunks,
    // which follow event waits on their input copies.
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    // Stream-K owners wait on peers with higher CTA indices, which never
    // wait themselves.  The grid is at most one CTA per SM (one CTA fits per
    // SM; cluster grids are sized to cudaOccupancyMaxActiveClusters), so every
    // peer gets an SM once the GPU has room, and the waits are bounded: a
    // peer that cannot run in time turns into GEMM_ERR_TIMEOUT, never a hang.
    cfg.attrs = attr;
    cfg.numAttrs = na;
    void* args[4] = {&p->tmA, &p->tmB, &p->tmC, &kp};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_status_t gemm_run_host(gemm_plan_t p, const void* hA, const void* hB, void* hC, void* dA,
                            void* dB, void* dC, void* workspace, gemm_stream_t stream) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (p->offline) return GEMM_ERR_NO_DEVICE;
    if (p->M == 0 || p->N == 0) return GEMM_OK;
    if (!hC || !dC || (p->K > 0 && (!hA || !hB || !dA || !dB))) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(p->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t a_bytes = (size_t)p->M * p->K * 2, b_bytes = (size_t)p->K * p->N * 2;
    const size_t c_bytes = (size_t)p->M * p->N * 2;
    int64_t rows = 0, cols = 0;
    int nr = 1, nc = 1;
    int blocks = host_grid(p, &rows, &cols, &nr, &nc);
    // the pipeline is a speed-up only: if its streams, events or sub-plans
    // cannot be made, run the serial path
    if (blocks > 1 && pipe_prepare(p, rows, cols) != GEMM_OK) blocks = 1;
    if (blocks <= 1) {
        if (p->K > 0) {
            if (cudaMemcpyAsync(dA, hA, a_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
                cudaMemcpyAsync(dB, hB, b_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
                return GEMM_ERR_CUDA;
        }
        gemm_status_t r = gemm_run(p, dA, dB, dC, workspace, stream);
        if (r != GEMM_OK) return r;
        if (cudaMemcpyAsync(hC, dC, c_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return GEMM_ERR_CUDA;
        return GEMM_OK;
    }
    // Pipelined over an nr x nc grid of blocks: row chunks of A and column
    // chunks of B are copied in on one internal stream, A_0, B_0, A_1, B_1, ...;
    // block (i, j) is computed on `stream` once A_i and B_j have arrived, in
    // the order their inputs complete, and copied out on a second internal
    // stream.  Entry and exit are ordered with the caller's stream by events.
    const bool a_col = p->layout_a == GEMM_COL_MAJOR, b_row = p->layout_b == GEMM_ROW_MAJOR;
    const char* ha = static_cast<const char*>(hA);
    const char* hb = static_cast<const char*>(hB);
    char* da = static_cast<char*>(dA);
    char* db = static_cast<char*>(dB);
    char* hc = static_cast<char*>(hC);
    char* dc = static_cast<char*>(dC);
    const size_t M2 = (size_t)p->M * 2, N2 = (size_t)p->N * 2, K2 = (size_t)p->K * 2;
#define PSM_CUDA(x) do { if ((x) != cudaSuccess) return GEMM_ERR_CUDA; } while (0)
    PSM_CUDA(cudaEventRecord(p->ev_start, st));
    PSM_CUDA(cudaStreamWaitEvent(p->h2d, p->ev_start, 0));
    PSM_CUDA(cudaStreamWaitEvent(p->d2h, p->ev_start, 0));
    for (int k = 0; k < std::max(nr, nc); ++k) {
        if (k < nr) {  // rows r0 .. r0+n-1 of A
            const int64_t r0 = (int64_t)k * rows, n = std::min(rows, p->M - r0);
            if (!a_col)
                PSM_CUDA(cudaMemcpyAsync(da + r0 * K2, ha + r0 * K2, n * K2, cudaMemcpyHostToDevice, p->h2d));
            else
                PSM_CUDA(cudaMemcpy2DAsync(da + r0 * 2, M2, ha + r0 * 2, M2, n * 2, (size_t)p->K,
                                           cudaMemcpyHostToDevice, p->h2d));
            PSM_CUDA(cudaEventRecord(p->ev_a[k], p->h2d));
        }
        if (k < nc) {  // columns c0 .. c0+n-1 of B
            const int64_t c0 = (int64_t)k * cols, n = std::min(cols, p->N - c0);
            if (!b_row)
                PSM_CUDA(cudaMemcpyAsync(db + c0 * K2, hb + c0 * K2, n * K2, cudaMemcpyHostToDevice, p->h2d));
            else
                PSM_CUDA(cudaMemcpy2DAsync(db + c0 * 2, N2, hb + c0 * 2, N2, n * 2, (size_t)p->K,
                                           cudaMemcpyHostToDevice, p->h2d));
            PSM_CUDA(cudaEventRecord(p->ev_b[k], p->h2d));
        }
    }
    // The sub-plans and this plan share `workspace`, each with its own flag
    // layout.  Each sub-plan clears the shared flag region before its first
    // block of this call; its later blocks (and blocks of the other
    // sub-plan that follow them) find flags left by earlier runs and rely on
    // the epoch tag: a post restarts a flag from another run at 1, and no
    // wait matches another run's value.  This plan clears its own flags
    // again on its next gemm_run.
    for (gemm_plan* sp : p->sub)
        if (sp) sp->flags_cleared_for = nullptr;
    p->flags_cleared_for = nullptr;
    int done = 0;
    for (int k = 0; k < std::max(nr, nc); ++k) {
        // blocks whose later input is A_k or B_k: (k, 0..k) then (0..k-1, k)
        for (int t = 0; t < 2 * k + 1; ++t) {
            const int i = t <= k ? k : t - k - 1, j = t <= k ? t : k;
            if (i >= nr || j >= nc) continue;
            const int64_t r0 = (int64_t)i * rows, c0 = (int64_t)j * cols;
            gemm_plan* sp = p->sub[2 * (i == nr - 1 && p->sub[2] ? 1 : 0) +
                                   (j == nc - 1 && (p->sub[1] || p->sub[3]) ? 1 : 0)];
            const void* a_blk = a_col ? (const void*)(da + r0 * 2) : (const void*)(da + r0 * K2);
            const void* b_blk = b_row ? (const void*)(db + c0 * 2) : (const void*)(db + c0 * K2);
            PSM_CUDA(cudaStreamWaitEvent(st, p->ev_a[i], 0));
            PSM_CUDA(cudaStreamWaitEvent(st, p->ev_b[j], 0));
            gemm_status_t r = run_impl(sp, a_blk, b_blk, dc + r0 * N2 + c0 * 2, workspace, stream, false);
            if (r != GEMM_OK) return r;
            PSM_CUDA(cudaEventRecord(p->ev_c[done], st));
            PSM_CUDA(cudaStreamWaitEvent(p->d2h, p->ev_c[done], 0));
            PSM_CUDA(cudaMemcpy2DAsync(hc + r0 * N2 + c0 * 2, N2, dc + r0 * N2 + c0 * 2, N2,
                                       (size_t)sp->N * 2, (size_t)sp->M, cudaMemcpyDeviceToHost, p->d2h));
            ++done;
        }
    }
    PSM_CUDA(cudaEventRecord(p->ev_done, p->d2h));
    PSM_CUDA(cudaStreamWaitEvent(st, p->ev_done, 0));
#undef PSM_CUDA
    return GEMM_OK;
}

gemm_status_t gemm_last_status(gemm_plan_t p, gemm_stream_t stream) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (p->offline) return GEMM_ERR_NO_DEVICE;
    DeviceGuard guard(p->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (h != STATUS_OK) {
        if (cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
        return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

gemm_status_t gemm_plan_units(gemm_plan_t p, int64_t cta, int32_t* units, int64_t max_units,
                              int64_t* n_units) {
    if (!p || !n_units || cta < 0 || cta >= p->ctas || max_units < 0 ||
        (max_units > 0 && !units))
        return GEMM_ERR_INVALID_ARG;
    const int32_t unit_cta = (int32_t)(cta / p->CM);  // both CTAs of a pair run the same units
    Sched hs = p->s;
    hs.raster_table = (p->opt_raster == 1 && p->raster_host) ? p->raster_host->data() : nullptr;
    Cursor cur;
    cursor_init(hs, unit_cta, cur);
    Unit u;
    int64_t n = 0;
    while (cursor_next(hs, unit_cta, cur, u)) {
        if (n < max_units) {
            int32_t* o = units + 5 * n;
            o[0] = u.tile;
            o[1] = u.k0;
            o[2] = u.k1;
            o[3] = u.role;
            o[4] = u.npeers;
        }
        ++n;
    }
    *n_units = n;
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_trace(gemm_plan_t p, void* device_buffer, size_t bytes) {
    if (!p || (device_buffer && ((uintptr_t)device_buffer & 7u))) return GEMM_ERR_INVALID_ARG;
    p->trace = reinterpret_cast<unsigned long long*>(device_buffer);
    p->trace_bytes = device_buffer ? bytes : 0;
    return GEMM_OK;
}

gemm_status_t gemm_plan_tile_coords(gemm_plan_t p, int64_t tile, int64_t* tile_m, int64_t* tile_n) {
    if (!p || !tile_m || !tile_n || tile < 0 || tile >= p->s.tiles) return GEMM_ERR_INVALID_ARG;
    int32_t tm, tn;
    Sched hs = p->s;
    hs.raster_table = (p->opt_raster == 1 && p->raster_host) ? p->raster_host->data() : nullptr;
    tile_coords(hs, (int32_t)tile, tm, tn);
    *tile_m = tm;
    *tile_n = tn;
    return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t p) {
    if (!p) return GEMM_OK;
    pipe_release(p);
    if (p->d_status && p->owns_status) cudaFree(p->d_status);
    if (p->raster_dev) cudaFree(p->raster_dev);
    delete p->raster_host;
    delete p;
    return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: alignment, stride or option not supported";
        case GEMM_ERR_WORKSPACE: return "GEMM_ERR_WORKSPACE: workspace missing or misaligned";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA runtime call failed";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch refused";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a bounded device wait expired";
        case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE: no sm_103 device for this plan";
    }
    return "GEMM_ERR_UNKNOWN";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc: for example a plug-in that runs inside
// a host framework which owns every byte of device memory and forbids
// allocation on its execution path, or a caller whose memory budget is fixed
// before the first product runs.  gemm_run_no_alloc serves them: instead of a
// caller-provided workspace, the Stream-K flags and partial tiles live in the
// fixed array below, which every GPU that loads this library holds until the
// process exits.  Plans whose workspace exceeds it are rejected.
//
// The array's name is a host-side stand-in in host code, not a device
// address, so the host looks up the real address once per device with
// cudaGetSymbolAddress, with that device current, on the first call for that
// device.  Every call shares the array and finds the previous call's data in
// it; calls that overlap on the GPU race on it.
static __device__ __align__(256) unsigned char psm_no_alloc_scratch[GEMM_NO_ALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_no_alloc_mu;
void* g_no_alloc_ptr[kMaxDevices];
}  // namespace

extern "C" gemm_status_t gemm_run_no_alloc(gemm_plan_t p, const void* A, const void* B, void* C,
                                           gemm_stream_t stream) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (p->offline) return GEMM_ERR_NO_DEVICE;
    if (p->ws_bytes > (size_t)GEMM_NO_ALLOC_SCRATCH_BYTES) return GEMM_ERR_WORKSPACE;
    if (p->ws_bytes == 0) return gemm_run(p, A, B, C, nullptr, stream);
    if (p->device < 0 || p->device >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        DeviceGuard guard(p->device);  // the look-up must run with the plan's device current
        if (!guard.ok) return GEMM_ERR_CUDA;
        std::lock_guard<std::mutex> lock(g_no_alloc_mu);
        if (!g_no_alloc_ptr[p->device]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, psm_no_alloc_scratch) != cudaSuccess || !ptr) {
                cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            g_no_alloc_ptr[p->device] = ptr;
        }
        scratch = g_no_alloc_ptr[p->device];
        // the flags left by an earlier call (possibly of another plan) are cleared
        // so this run starts from zero; the partial slots are always written
        // before they are read
        if (cudaMemsetAsync(scratch, 0, p->ws_flag_bytes, reinterpret_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    return gemm_run(p, A, B, C, scratch, stream);
}
