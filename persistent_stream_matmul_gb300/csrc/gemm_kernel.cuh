// sm_103a GEMM kernel: C = A * B, fp16/bf16 in, fp32 accumulation in tensor
// memory, fp16/bf16 out.  One kernel serves the data-parallel, persistent and
// Stream-K schedules; the tile scheduler (sched.cuh) tells every CTA which
// work units (tile, k-range, role) it runs.
//
// Clusters (CM = 2): the two CTAs of a cluster run the same scheduled unit on
// the two 128-row halves of a 256-row tile, so they need the same B tile.
// Each CTA loads its own A and half of B; L2-to-SM traffic per CTA drops from
// A + B to A + B/2 per k-slice.  Two ways to use the halves:
//   PAIR_MMA   one thread of the first CTA issues tcgen05.mma.cta_group::2
//              (256 x BN) over both CTAs' shared memory, each CTA keeping only
//              its half of B (a deeper ring); both CTAs' copies complete on the
//              first CTA's barriers, and one multicast commit frees both rings.
//   otherwise  each CTA multicasts its half of B into both rings and runs its
//              own 128 x BN MMA; a stage's empty barrier counts the commits of
//              both CTAs, so neither refills a stage the other still reads.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: one lane fills a STAGES-deep ring of A/B tiles
//               in shared memory (128-byte swizzle), guarded by full/empty
//               mbarriers.
//   warp 1      allocates tensor memory (two accumulators of 128 x BN fp32);
//               one lane issues tcgen05.mma (128 x BN x 16 each) and commits
//               to the ring's empty barriers and to the accumulator barriers.
//   warps 2-5   epilogue: drain an accumulator (tcgen05.ld) while the MMA
//               fills the other one.  FULL unit: round once to the output
//               type and store C with 16-byte vector stores.  PEER unit
//               (Stream-K, not holding k-iteration 0): store the fp32 partial
//               to this CTA's workspace slot, then post the tile's flag.
//               OWNER unit (holds k-iteration 0): wait until all the tile's
//               peers have posted, add their partials in ascending k, round
//               once, store C.  At a CTA's last unit the ring is idle: the
//               peers' partials are copied into it in one round trip, and C
//               is staged there and written as whole rows.
//               CLUSTER_PART unit (cluster split-K): the fp32 partial goes
//               to this CTA's idle ring; once every CTA of the cluster has
//               signalled its own, each adds all parts of its slice of the
//               tile's columns, read through distributed shared memory in
//               ascending part order, rounds once and stores C.
//
// Sources: the HF post "naive vs persistent matmul" (tile per thread-block,
// persistent thread-blocks, warp specialisation and double buffering named
// as the tricks that reach peak); the GitHub issue "Stream-k matmul
// implementation very slow ..." (the Stream-K split and the fixup, whose
// "scratchpad + barrier" form is used here instead of atomic adds).
//
// Every wait is bounded: a pipeline wait that runs out sets the CTA's abort
// flag and the device status word, and all roles leave their loops; an owner
// whose peers do not post in time skips the tile's store and records a
// timeout.  Nothing traps.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sched.cuh"

namespace psm {

constexpr int BM = 128;              // tile rows (TMEM lanes)
constexpr int BK = 64;               // k-slice: 64 x 2 B = one 128-byte swizzle row
constexpr int UMMA_K = 16;           // k of one tcgen05.mma kind::f16
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;         // first epilogue warp
constexpr int EPI_THREADS = 128;
constexpr int SW_ATOM_BYTES = 1024;  // 8 rows x 128 B
constexpr int MN_CHUNK_BYTES = 64 * BK * 2;  // one 64-element-wide MN-major box (8 KB)

enum : int { STATUS_OK = 0, STATUS_FLAG_TIMEOUT = 1, STATUS_PIPE_TIMEOUT = 2 };
enum : uint32_t { BAR_EPI_SYNC = 1, BAR_EPI_VOTE = 2 };  // named barriers (0 = __syncthreads)

template <bool V>
struct BoolConst {
    static constexpr bool value = V;
};

// AROWS: rows of A loaded per stage.  128 normally.  64 when M <= 64: the
// MMA still reads 128 rows, and rows 64-127 alias the first bytes of the
// stage's B tile, so those accumulator rows hold garbage that is never stored
// (each output row depends only on its own row of A); the smaller stage lets
// the ring hold more B in flight.
template <int BN, int AROWS = 128, bool PAIR_MMA = false>
struct Cfg {
    static constexpr int A_STAGE_BYTES = AROWS * BK * 2;
    // a pair MMA keeps only this CTA's half of the B tile in its ring
    static constexpr int B_STAGE_BYTES = (PAIR_MMA ? BN / 2 : BN) * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    // Ring of up to 224 KB (the CTA may hold 227 KB; barriers and alignment
    // take the rest), at most 12 stages.  Pair-MMA kernels also write C
    // through tensor copies from a staging area of 4 KB per epilogue warp
    // (32 rows x 128 bytes, one 64-column box) after the ring, taken from the
    // same budget.  Stages: 4 at BN=256, 7 at BN=128, 9 with half-height A at
    // BN=128 and 5 with it at BN=256; with a pair MMA, 6 at BN=256 and 8 at
    // BN=128.
    static constexpr int EPI_STAGE_BYTES = PAIR_MMA ? 4 * 32 * 128 : 0;
    static constexpr int STAGES_FIT = (224 * 1024 - EPI_STAGE_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
    static constexpr int TMEM_COLS = 2 * BN;  // two accumulators; 256 or 512
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
    static_assert(AROWS == 128 || AROWS == 64, "rows of A per stage");
    static_assert(AROWS == 128 || A_STAGE_BYTES + B_STAGE_BYTES >= BM * BK * 2,
                  "the MMA's 128-row read of A must stay inside the stage");
    static_assert((2 * STAGES + 7) * 8 + 8 <= BAR_BYTES, "barrier area");
};

struct KParams {
    Sched s;
    int32_t M, N, K;
    int32_t ldc;                 // elements between rows of C (N, or more for a block of a wider C)
    void* C;
    float* partials;             // Stream-K: grid slots of BM x BN fp32
    unsigned long long* flags;   // Stream-K: one flag per split tile
    int* status;                 // device status word (first error wins)
    uint32_t idesc;
    uint32_t epoch;              // run number tagged into the flags
    int32_t a_mn, b_mn;          // operand major-ness: 0 = K-major, 1 = MN-major
    int32_t inject_skip_cta;     // test hook, -1 = off
    uint64_t wait_limit_ns;      // owner's wait for its peers
    uint64_t pipe_limit_ns;      // any wait inside the CTA's own pipeline
    unsigned long long* trace;   // optional: TRACE_N stamps per CTA, or null
    int32_t early_prefetch;      // k-blocks of the first unit brought into L2 before the wait
    int32_t c_tma;               // 1: whole tiles store C through tensor copies (tmC)
};

// Per-CTA trace stamps: nanoseconds of %globaltimer at the start of the CTA,
// prologue done (after the wait for earlier grids), last copy issued by the
// producer, CTA end (all epilogue stores issued); then the SM's %clock64 at
// the start and at the end, so that (cycles / nanoseconds) is the SM clock
// the CTA ran at.
enum : int {
    TRACE_START = 0, TRACE_READY = 1, TRACE_LOADS_DONE = 2, TRACE_END = 3,
    TRACE_CLK_START = 4, TRACE_CLK_END = 5, TRACE_N = 6
};

__device__ __forceinline__ void record_status(int* status, int code) {
    atomicCAS(status, 0, code);
}

// Post one peer contribution to a split tile's flag.  The flag holds
// (epoch << 32) | posts; a value from an older run is restarted at 1.
__device__ __forceinline__ void post_flag(unsigned long long* f, uint32_t epoch) {
    uint64_t cur = *reinterpret_cast<volatile unsigned long long*>(f);
#pragma unroll 1
    for (int tries = 0; tries < (1 << 20); ++tries) {
        uint64_t want = ((uint32_t)(cur >> 32) == epoch) ? cur + 1
                                                         : (((uint64_t)epoch << 32) | 1ull);
        uint64_t prev = atom_cas_release_u64(f, cur, want);
        if (prev == cur) return;
        cur = prev;
    }
}

__device__ __forceinline__ bool wait_flag(const unsigned long long* f, uint64_t target,
                                          uint64_t limit_ns) {
    if (ld_acquire_u64(f) == target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i) {
            if (ld_acquire_u64(f) == target) return true;
            __nanosleep(32);
        }
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// AND of a predicate over the 128 epilogue threads.
__device__ __forceinline__ bool epi_vote_all(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"((uint32_t)BAR_EPI_VOTE), "r"((uint32_t)EPI_THREADS)
        : "memory");
    return out != 0;
}

template <bool OUT_BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b);

// Cluster split-K: this CTA's slice of the tile, columns [part * BN / KC,
// (part + 1) * BN / KC) of rows [0, rows), as 16-byte units of 4 fp32.  Every
// CTA of the cluster holds its own part of the whole tile in its shared
// memory at `sbase`, row r at r * BN * 4 bytes with unit u at
// ((u ^ (r & 7)) * 16).  Each unit of the slice is the sum of the KC parts in
// ascending part (= k) order, ((P0 + P1) + P2) + ..., in fp32, rounded once
// and stored to C (tile origin `ctile`, row stride ldc elements, first column
// col0).  The parts of BATCH units are loaded before any is added, so 16
// loads are in flight per thread instead of one round trip per unit.
template <int KC, int BN, bool OUT_BF16>
__device__ __forceinline__ void cluster_reduce_slice(uint32_t sbase, int part, int rows, int et,
                                                     uint8_t* ctile, int ldc, int col0, int N) {
    constexpr int W4 = BN / 4 / KC;     // units of the slice in one row
    constexpr int BATCH = 16 / KC;      // units per thread per round
    constexpr uint32_t ROW_BYTES = (uint32_t)BN * 4;
    const int total = rows * W4;
#pragma unroll 1
    for (int base = et; base < total; base += EPI_THREADS * BATCH) {
        float4 x[BATCH][KC];
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int idx = base + b * EPI_THREADS;
            if (idx < total) {
                const int row = idx / W4;
                const int gu = part * W4 + idx % W4;
                const uint32_t a = sbase + (uint32_t)row * ROW_BYTES + (uint32_t)((gu ^ (row & 7)) * 16);
#pragma unroll
                for (int q = 0; q < KC; ++q)
                    x[b][q] = q == part ? ld_shared_f4(a) : ld_cluster_f4(mapa_shared(a, (uint32_t)q));
            }
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int idx = base + b * EPI_THREADS;
            if (idx < total) {
                const int row = idx / W4;
                const int col = col0 + (part * W4 + idx % W4) * 4;
                float4 acc = x[b][0];
#pragma unroll
                for (int q = 1; q < KC; ++q) {
                    acc.x += x[b][q].x;
                    acc.y += x[b][q].y;
                    acc.z += x[b][q].z;
                    acc.w += x[b][q].w;
                }
                if (col < N)
                    st_u2(ctile + ((size_t)row * ldc + col) * 2, pack2<OUT_BF16>(acc.x, acc.y),
                          pack2<OUT_BF16>(acc.z, acc.w));
            }
        }
    }
}

// Cluster split-K exchange by bulk copies, when the ring holds both a staged
// partial and the slots for the other parts (2 * AROWS * BN * 4 bytes).  CTA
// `part` owns columns [part * BN / KC, (part + 1) * BN / KC) of the tile.
//  1. Its ring is idle (this accumulator is ready): tell the other CTAs they
//     may copy into it, and arm this CTA's receive barrier for their bytes.
//  2. Stage the partial slice by slice (slice q at q * SLOT: row r at
//     r * W * 4, 16-byte units XOR-swizzled by row), so each slice is one
//     contiguous block.
//  3. Once the other CTAs may be written, one thread bulk-copies each
//     foreign slice into its owner's slot for this part (the copy engine,
//     completing on the owner's barrier in bytes).
//  4. Wait for this CTA's slots, then sum its slice in ascending part (= k)
//     order, ((P0 + P1) + P2) + ..., in fp32, round once and store C.
// Every wait is bounded; one that runs out records a timeout and the CTA
// stores nothing.  skip_copies (test hook) withholds step 3.
template <int KC, int BN, int AROWS, bool OUT_BF16>
__device__ __forceinline__ void cluster_exchange_bulk(uint32_t ring, uint32_t free_bar, uint32_t recv_bar,
                                                      int part, uint32_t tbase, int row, bool row_ok,
                                                      int rows, int et, bool empty, bool skip_copies,
                                                      uint64_t limit_ns, int* status, uint8_t* ctile,
                                                      int ldc, int col0, int N) {
    constexpr int W = BN / KC;                   // columns of a slice
    constexpr int U = W / 4;                     // 16-byte units in a slice row
    constexpr int SW = (U < 8 ? U : 8) - 1;      // swizzle mask
    constexpr uint32_t SLOT = (uint32_t)AROWS * W * 4;
    constexpr uint32_t RECV = (uint32_t)KC * SLOT;  // slots after the staged partial
    static_assert(U >= 4 && (U & (U - 1)) == 0, "slice rows of 4, 8, 16 or 32 units");
    const uint32_t bytes = (uint32_t)rows * W * 4;  // a slice's valid rows, a multiple of 16
    // 1. this ring is free: the other parts may copy into its slots
    fence_proxy_async_smem();  // the ring was last used by the async proxy
    named_bar_sync(BAR_EPI_SYNC, EPI_THREADS);
    if (et == 0) {
        mbar_arrive_expect_tx(recv_bar, (uint32_t)(KC - 1) * bytes);
#pragma unroll
        for (int q = 0; q < KC; ++q)
            if (q != part) mbar_arrive_cluster(mapa_shared(free_bar, (uint32_t)q));
    }
    // 2. stage the partial, slice by slice
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + j * 32, r);
        if (row_ok) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int gu = j * 8 + v;
                const int q = gu / U, u = gu % U;
                st_shared_u4(ring + (uint32_t)q * SLOT + (uint32_t)row * (W * 4) + (uint32_t)((u ^ (row & SW)) * 16),
                             empty ? 0u : r[4 * v], empty ? 0u : r[4 * v + 1], empty ? 0u : r[4 * v + 2],
                             empty ? 0u : r[4 * v + 3]);
            }
        }
    }
    fence_proxy_async_smem();  // the staged bytes, for the copy engine
    named_bar_sync(BAR_EPI_SYNC, EPI_THREADS);
    // 3. copy the foreign slices once their owners may be written
    bool sent = false;
    if (et == 0) {
        const bool may = mbar_wait_acq_cluster(free_bar, 0, limit_ns);
        if (!may) record_status(status, STATUS_FLAG_TIMEOUT);
        if (may && !skip_copies) {
#pragma unroll
            for (int q = 0; q < KC; ++q)
                if (q != part)
                    bulk_copy_to_cluster(mapa_shared(ring + RECV + (uint32_t)part * SLOT, (uint32_t)q),
                                         ring + (uint32_t)q * SLOT, bytes,
                                         mapa_shared(recv_bar, (uint32_t)q));
            bulk_commit_group();
            sent = true;
        }
    }
    // 4. this CTA's slots, then its slice
    const bool got = epi_vote_all(mbar_wait_acq_cluster(recv_bar, 0, limit_ns));
    if (!got) {
        if (et == 0) record_status(status, STATUS_FLAG_TIMEOUT);
    } else {
        constexpr int BATCH = 16 / KC;
        const int total = rows * U;
#pragma unroll 1
        for (int base = et; base < total; base += EPI_THREADS * BATCH) {
            float4 x[BATCH][KC];
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int idx = base + b * EPI_THREADS;
                if (idx < total) {
                    const int rr = idx / U, u = idx % U;
                    const uint32_t off = (uint32_t)rr * (W * 4) + (uint32_t)((u ^ (rr & SW)) * 16);
#pragma unroll
                    for (int s = 0; s < KC; ++s)
                        x[b][s] = ld_shared_f4(s == part ? ring + (uint32_t)part * SLOT + off
                                                         : ring + RECV + (uint32_t)s * SLOT + off);
                }
            }
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int idx = base + b * EPI_THREADS;
                if (idx < total) {
                    const int rr = idx / U;
                    const int col = col0 + (part * U + idx % U) * 4;
                    float4 acc = x[b][0];
#pragma unroll
                    for (int s = 1; s < KC; ++s) {
                        acc.x += x[b][s].x;
                        acc.y += x[b][s].y;
                        acc.z += x[b][s].z;
                        acc.w += x[b][s].w;
                    }
                    if (col < N)
                        st_u2(ctile + ((size_t)rr * ldc + col) * 2, pack2<OUT_BF16>(acc.x, acc.y),
                              pack2<OUT_BF16>(acc.z, acc.w));
                }
            }
        }
    }
    // the copies out of this CTA's ring have landed before it may be released
    if (sent) bulk_wait_group_0();
}

template <bool OUT_BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (OUT_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// KCL: cluster split-K; the CTAs of a cluster (p.s.kc of them, along x) are
// the k-parts of one tile and reduce through distributed shared memory.
template <int BN, bool OUT_BF16, int CM, int AROWS = 128, bool PAIR_MMA = false, bool KCL = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ KParams p) {
    using Cf = Cfg<BN, AROWS, PAIR_MMA>;
    static_assert(!PAIR_MMA || CM == 2, "a pair MMA needs a 2-CTA cluster");
    static_assert(AROWS == 128 || CM == 1 || PAIR_MMA, "half-height A: no multicast clusters");
    static_assert(BN >= 128 || CM == 1, "64-wide tiles only without clusters");
    constexpr int STAGES = Cf::STAGES;
    static_assert(CM == 1 || CM == 2, "cluster size");
    static_assert(!KCL || (CM == 1 && !PAIR_MMA && BN >= 128), "cluster split-K: 1-CTA MMAs");
    constexpr uint16_t PAIR_MASK = 0x3;
    extern __shared__ uint8_t smem_raw[];

    // 1024-byte aligned base: the 128-byte swizzle pattern repeats every 1 KB
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    const uint32_t epi_stage = sbase + STAGES * Cf::STAGE_BYTES;  // C boxes (pair MMA)
    uint8_t* bar_area = smem_raw + pad + STAGES * Cf::STAGE_BYTES + Cf::EPI_STAGE_BYTES;
    const uint32_t bar_base = epi_stage + Cf::EPI_STAGE_BYTES;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar_base + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bar_base + 8u * (2 * STAGES + 4);
    // cluster split-K: the other parts' signals, and the bytes of their slices
    const uint32_t parts_bar = bar_base + 8u * (2 * STAGES + 5);
    const uint32_t recv_bar = bar_base + 8u * (2 * STAGES + 6);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * STAGES + 7));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (2 * STAGES + 7) + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;                      // workspace slot of this CTA
    const uint64_t t_start = globaltimer_ns();
    const uint64_t c_start = sm_clock64();
    const int unit_cta = blockIdx.x / CM;            // index the scheduler knows
    const int rank = CM == 2 ? (int)cluster_ctarank() : 0;

    if (threadIdx.x == 0) {
        // pair MMA: the first CTA's full barriers count both CTAs' copies, one
        // multicast commit frees a stage in both CTAs, and the first CTA's
        // accumulator-empty barriers count the epilogue warps of both
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), PAIR_MMA ? 1 : CM);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), (PAIR_MMA ? 2 : 1) * EPI_THREADS / 32);
        }
        mbar_init(done_bar, 1);
        // one release-arrive from each other CTA of the cluster
        if constexpr (KCL) {
            mbar_init(parts_bar, (uint32_t)(p.s.kc > 1 ? p.s.kc - 1 : 1));
            mbar_init(recv_bar, 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        if constexpr (PAIR_MMA) {
            tmem_alloc_pair(smem_addr(tmem_slot), Cf::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(tmem_slot), Cf::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    if constexpr (CM == 2 || KCL) {
        // the other CTAs' barriers exist before anything is multicast or
        // arrives remotely
        cluster_sync_all();
    } else {
        __syncthreads();
    }
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // Everything above touches only this CTA's shared and tensor memory, so
    // it may overlap the previous kernel in the stream; global memory (A, B,
    // C, workspace, status) is touched only after that kernel has finished.
    // The one exception is an L2 prefetch of the operands of this CTA's first
    // unit (GEMM_OPT_EARLY_PREFETCH): it brings lines into L2 without
    // reading them into the CTA, and L2 is the point of coherence, so a write
    // by the previous kernel to the same lines still lands before any read
    // made after the wait.  It uses the DRAM time of the previous kernel's
    // tail, for the CTAs that start on SMs that kernel left idle.
    if (p.early_prefetch > 0 && warp == 0 && lane == 0) {
        Cursor cur;
        cursor_init(p.s, unit_cta, cur);
        Unit u;
        if (cursor_next(p.s, unit_cta, cur, u)) {
            const int m0 = (u.tm * CM + rank) * BM, n0 = u.tn * BN;
            const int nk = min(u.k1 - u.k0, p.early_prefetch);
            for (int i = 0; i < nk; ++i) {
                const int k_el = unit_kblock(p.s, u.tile, u.k0, u.k1, i) * BK;
                if (!p.b_mn) {
                    tma_prefetch_l2_2d(&tmB, k_el, n0 + rank * (BN / CM));
                } else {
#pragma unroll 1
                    for (int c = rank * (BN / 64) / CM; c < (rank + 1) * (BN / 64) / CM; ++c)
                        tma_prefetch_l2_2d(&tmB, n0 + 64 * c, k_el);
                }
                if (!p.a_mn) {
                    tma_prefetch_l2_2d(&tmA, k_el, m0);
                } else {
#pragma unroll 1
                    for (int c = 0; c < AROWS / 64; ++c) tma_prefetch_l2_2d(&tmA, m0 + 64 * c, k_el);
                }
            }
        }
    }
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        grid_launch_dependents();
        if (p.trace) {
            p.trace[(size_t)cta * TRACE_N + TRACE_START] = t_start;
            p.trace[(size_t)cta * TRACE_N + TRACE_READY] = globaltimer_ns();
        }
    }

    auto fail_pipe = [&]() {
        *abort_flag = 1;
        record_status(p.status, STATUS_PIPE_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop and takes every branch together (waits
        // are voted); one elected lane issues the copies.  With the loop run
        // by lane 0 alone, its values were not warp-uniform and each copy took
        // ~130 cycles to issue, on the ring's critical path: the warp-wide
        // form took ~9 % off the SM cycles of a large square product.
        {
            // With a single row of tiles every B tile is read exactly once:
            // let it leave L2 first and keep the small, shared A resident.
            // Otherwise the copies carry no L2 policy at all (the cache-hint
            // form measured ~1.5 % slower on a large square product).  The
            // choice is a compile-time constant of the loop below: a run-time
            // branch between the two copy forms made that loop ~7 % slower.
            const bool b_once = p.s.tiles_m == 1;
            const uint64_t pol_a = b_once ? l2_policy_evict_last() : l2_policy_evict_normal();
            const uint64_t policy = b_once ? l2_policy_evict_first() : l2_policy_evict_normal();
            Cursor cur;
            cursor_init(p.s, unit_cta, cur);
            Unit u;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;  // per-stage bit masks
            bool ok = true;
            // pair MMA: the first CTA's full barriers, as shared::cluster
            // addresses (consecutive like the local ones)
            const uint32_t full0_c = PAIR_MMA ? mapa_shared(full_bar(0), 0) : 0u;
            auto produce = [&](auto hint_tag) {
                constexpr bool HINT = decltype(hint_tag)::value;
                while (ok && cursor_next(p.s, unit_cta, cur, u)) {
                    const int m0 = (u.tm * CM + rank) * BM, n0 = u.tn * BN;
                    const int nk = u.k1 - u.k0;
                    // Per-unit work stays out of the k-loop: whether the unit's
                    // k-blocks are rotated, and the abort check.  The loop is on
                    // the ring's critical path (a stage is refilled as soon as
                    // it is released); with these in it, and the peer barrier
                    // address recomputed every k-block, the tensor pipe idled
                    // ~9 % more of its cycles on a large square product.
                    const bool rot_unit = p.s.k_rotate && u.k0 == 0 && u.k1 == p.s.ipt;
                    if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
                    // L2 prefetch of B, l2_prefetch k-blocks ahead of the loads: keeps
                    // DRAM busy beyond what the shared-memory ring can hold in flight
                    const int pf = p.s.l2_prefetch;
                    auto prefetch_b = [&](int step) {
                        const int kp = unit_kblock(p.s, u.tile, u.k0, u.k1, step) * BK;
                        if (!p.b_mn) {
                            tma_prefetch_l2_2d(&tmB, kp, n0 + rank * (BN / CM));
                        } else {
#pragma unroll
                            for (int c = rank * (BN / 64) / CM; c < (rank + 1) * (BN / 64) / CM; ++c)
                                tma_prefetch_l2_2d(&tmB, n0 + 64 * c, kp);
                        }
                    };
                    if (lane == 0)
                        for (int i = 0; i < pf && i < nk; ++i) prefetch_b(i);
                    for (int i = 0; i < nk; ++i) {
                        const int kb = rot_unit ? unit_kblock(p.s, u.tile, u.k0, u.k1, i) : u.k0 + i;
                        if (pf > 0 && i + pf < nk && lane == 0) prefetch_b(i + pf);
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(empty_bar(stage), phase ^ 1u, p.pipe_limit_ns))) {
                            if (lane == 0) fail_pipe();
                            ok = false;
                            break;
                        }
                        if (elect_one()) {
                            const uint32_t fb = full_bar(stage);
                            const uint32_t sa = sbase + stage * Cf::STAGE_BYTES;
                            const uint32_t sb = sa + Cf::A_STAGE_BYTES;
                            const int k_el = kb * BK;
                            if constexpr (PAIR_MMA) {
                                // both CTAs' copies complete on the first CTA's barrier
                                const uint32_t fbc = full0_c + 8u * (uint32_t)stage;
                                if (rank == 0) mbar_arrive_expect_tx(fb, 2 * Cf::STAGE_BYTES);
                                if (!p.a_mn) {
                                    tma_load_2d_pair(sa, &tmA, fbc, k_el, m0, HINT, pol_a);  // AROWS rows
                                } else {
#pragma unroll
                                    for (int c = 0; c < AROWS / 64; ++c)
                                        tma_load_2d_pair(sa + c * MN_CHUNK_BYTES, &tmA, fbc, m0 + 64 * c,
                                                         k_el, HINT, pol_a);
                                }
                                const int nb = n0 + rank * (BN / 2);  // this CTA's half of B
                                if (!p.b_mn) {
                                    tma_load_2d_pair(sb, &tmB, fbc, k_el, nb, HINT, policy);
                                } else {
#pragma unroll
                                    for (int c = 0; c < BN / 128; ++c)
                                        tma_load_2d_pair(sb + c * MN_CHUNK_BYTES, &tmB, fbc, nb + 64 * c,
                                                         k_el, HINT, policy);
                                }
                            } else {
                            mbar_arrive_expect_tx(fb, Cf::STAGE_BYTES);
                            if (!p.a_mn) {
                                tma_load_2d(sa, &tmA, fb, k_el, m0, HINT, pol_a);  // box of AROWS rows
                            } else {
#pragma unroll
                                for (int c = 0; c < AROWS / 64; ++c)
                                    tma_load_2d(sa + c * MN_CHUNK_BYTES, &tmA, fb, m0 + 64 * c, k_el, HINT,
                                                pol_a);
                            }
                            if constexpr (CM == 1) {
                                if (!p.b_mn) {
                                    tma_load_2d(sb, &tmB, fb, k_el, n0, HINT, policy);
                                } else {
#pragma unroll
                                    for (int c = 0; c < BN / 64; ++c)
                                        tma_load_2d(sb + c * MN_CHUNK_BYTES, &tmB, fb, n0 + 64 * c, k_el, HINT,
                                                    policy);
                                }
                            } else {
                                // this CTA's half of B, into both CTAs of the pair
                                if (!p.b_mn) {
                                    const int half = BN / 2;  // rows of the K-major box
                                    tma_load_2d_multicast(sb + rank * half * 128, &tmB, fb, k_el,
                                                          n0 + rank * half, PAIR_MASK, HINT, policy);
                                } else {
#pragma unroll
                                    for (int c = rank * (BN / 128); c < (rank + 1) * (BN / 128); ++c)
                                        tma_load_2d_multicast(sb + c * MN_CHUNK_BYTES, &tmB, fb,
                                                              n0 + 64 * c, k_el, PAIR_MASK, HINT, policy);
                                }
                            }
                            }  // not a pair MMA
                        }
                        __syncwarp();
                        filled |= 1u << stage;
                        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            };
            if (b_once)
                produce(BoolConst<true>{});
            else
                produce(BoolConst<false>{});
            if (p.trace && lane == 0) p.trace[(size_t)cta * TRACE_N + TRACE_LOADS_DONE] = globaltimer_ns();
            // before the CTA (or its peer) exits: every copy into this CTA has
            // landed, and every MMA that reads this CTA's ring (the peer's too)
            // has released it
            for (int s = 0; s < STAGES; ++s)
                if (filled & (1u << s)) {
                    // (pair MMA: the second CTA's copies complete on the first
                    // CTA's barrier, so it waits for the stage's release alone)
                    if (!PAIR_MMA || rank == 0)
                        mbar_wait(full_bar(s), (fill_parity >> s) & 1u, p.pipe_limit_ns);
                    mbar_wait(empty_bar(s), (fill_parity >> s) & 1u, p.pipe_limit_ns);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // (pair MMA: the first CTA of the pair issues for both)
        // The whole warp runs the loop and takes every branch together (waits
        // are voted); one elected lane issues the MMAs and commits.  Run by
        // lane 0 alone, the loop's values are not warp-uniform and each
        // tcgen05 issue costs more: the warp-wide form took ~2 % off the SM
        // cycles of a large square product, on top of the producer's gain.
        if (!PAIR_MMA || rank == 0) {
            Cursor cur;
            cursor_init(p.s, unit_cta, cur);
            Unit u;
            int stage = 0;
            uint32_t phase = 0, iter = 0;
            bool ok = true;
            // Descriptors of stage 0's A and B tiles and the step of one
            // 16-element k-slice, computed once: the loop below only adds
            // offsets (the 14-bit address field cannot carry, the shared
            // window is below 256 KB).  The issue loop must stay lean: with
            // the descriptors rebuilt from kernel parameters for every MMA
            // (and reloaded after each one, the MMA asm clobbering memory),
            // and the abort flag read every k-block, the tensor pipe idled
            // ~10 % of the time even with no copies to wait for.
            //   K-major: a k-slice is 32 bytes along the swizzled row.
            //   MN-major: 16 k-rows of 128 bytes.
            const uint64_t a_desc0 =
                smem_desc_sw128(sbase, p.a_mn ? MN_CHUNK_BYTES : 16, SW_ATOM_BYTES);
            const uint64_t b_desc0 =
                smem_desc_sw128(sbase + Cf::A_STAGE_BYTES, p.b_mn ? MN_CHUNK_BYTES : 16, SW_ATOM_BYTES);
            const uint64_t a_kstep = p.a_mn ? (16 * 128) >> 4 : (UMMA_K * 2) >> 4;
            const uint64_t b_kstep = p.b_mn ? (16 * 128) >> 4 : (UMMA_K * 2) >> 4;
            const uint32_t idesc = p.idesc;
            while (ok && cursor_next(p.s, unit_cta, cur, u)) {
                const int buf = iter & 1;
                const bool got_t =
                    __all_sync(0xffffffffu, mbar_wait(tempty_bar(buf), ((iter >> 1) & 1u) ^ 1u, p.pipe_limit_ns));
                if (!got_t) {
                    if (lane == 0) fail_pipe();
                    break;
                }
                if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int i = 0; i < u.k1 - u.k0; ++i) {
                    if (!__all_sync(0xffffffffu, mbar_wait(full_bar(stage), phase, p.pipe_limit_ns))) {
                        if (lane == 0) fail_pipe();
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const bool leader = elect_one();
                    const uint64_t off = (uint64_t)((uint32_t)(stage * Cf::STAGE_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t adesc = a_desc0 + off + (uint64_t)kk * a_kstep;
                        const uint64_t bdesc = b_desc0 + off + (uint64_t)kk * b_kstep;
                        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                        if (leader) {
                            if constexpr (PAIR_MMA)
                                mma_f16_ss_pair(d_tmem, adesc, bdesc, idesc, acc);
                            else
                                mma_f16_ss(d_tmem, adesc, bdesc, idesc, acc);
                        }
                    }
                    if (leader) {
                        if constexpr (PAIR_MMA)
                            mma_commit_pair_multicast(empty_bar(stage), PAIR_MASK);  // frees both rings
                        else if constexpr (CM == 2)
                            mma_commit_multicast(empty_bar(stage), PAIR_MASK);  // both halves of B were read
                        else
                            mma_commit(empty_bar(stage));
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (elect_one()) {
                    if constexpr (PAIR_MMA)
                        mma_commit_pair_multicast(tfull_bar(buf), PAIR_MASK);  // both halves of D ready
                    else
                        mma_commit(tfull_bar(buf));
                }
                __syncwarp();
                ++iter;
            }
            // all MMAs the warp issued are complete before TMEM is freed
            __syncwarp();
            if (elect_one()) {
                if constexpr (PAIR_MMA)
                    mma_commit_pair_multicast(done_bar, 0x1);
                else
                    mma_commit(done_bar);
            }
            __syncwarp();
            mbar_wait(done_bar, 0, p.pipe_limit_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;              // TMEM lanes this warp may read: 32q .. 32q+31
        const int row_in_tile = q * 32 + lane;
        const int et = threadIdx.x - EPI_WARP0 * 32;
        Cursor cur;
        cursor_init(p.s, unit_cta, cur);
        Unit u;
        uint32_t iter = 0;
        while (cursor_next(p.s, unit_cta, cur, u)) {
            const int buf = iter & 1;
            bool ok = mbar_wait(tfull_bar(buf), (iter >> 1) & 1u, p.pipe_limit_ns) && !*abort_flag;
            if (!epi_vote_all(ok)) {
                if (et == 0) fail_pipe();
                break;
            }
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
            const int tm = u.tm * CM + rank;  // this CTA's 128-row tile
            const int rows_valid = min(BM, p.M - tm * BM);
            const int row = tm * BM + row_in_tile;
            const bool row_ok = row_in_tile < rows_valid;

            if constexpr (KCL && AROWS == 64) {
                // every unit of a cluster split-K plan is a CLUSTER_PART, and
                // the CTA's only unit.  With half-height A stages (M <= 64) the
                // ring holds the staged partial and the slots for the other
                // parts: exchange by bulk copies.  (Paired bursts: 1.3 % faster
                // on 64 x 8192 x 8192 and 3.9 % on 16 x 1024 x 16384 than the
                // pull below; on 128 x 4096 x 4096, with full-height tiles,
                // 1.8 % slower, so full-height tiles keep the pull.)
                static_assert(2u * AROWS * BN * 4 <= (uint32_t)STAGES * Cf::STAGE_BYTES,
                              "the staged partial and the slots fit the ring");
                const int part = (int)cluster_ctarank();  // = u.slot: CTA c is part c mod kc
                const bool empty = u.k1 <= u.k0;
                const bool skip = cta == p.inject_skip_cta;
                uint8_t* ctile = reinterpret_cast<uint8_t*>(p.C) + (size_t)tm * BM * p.ldc * 2;
                const int col0 = u.tn * BN;
                if (p.s.kc == 2)
                    cluster_exchange_bulk<2, BN, AROWS, OUT_BF16>(sbase, parts_bar, recv_bar, part, tbase,
                                                                  row_in_tile, row_ok, rows_valid, et, empty,
                                                                  skip, p.wait_limit_ns, p.status, ctile,
                                                                  p.ldc, col0, p.N);
                else if (p.s.kc == 4)
                    cluster_exchange_bulk<4, BN, AROWS, OUT_BF16>(sbase, parts_bar, recv_bar, part, tbase,
                                                                  row_in_tile, row_ok, rows_valid, et, empty,
                                                                  skip, p.wait_limit_ns, p.status, ctile,
                                                                  p.ldc, col0, p.N);
                else
                    cluster_exchange_bulk<8, BN, AROWS, OUT_BF16>(sbase, parts_bar, recv_bar, part, tbase,
                                                                  row_in_tile, row_ok, rows_valid, et, empty,
                                                                  skip, p.wait_limit_ns, p.status, ctile,
                                                                  p.ldc, col0, p.N);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(buf));
            } else if constexpr (KCL) {
                // every unit of a cluster split-K plan is a CLUSTER_PART
                // The CTA's only unit: its ring is idle (every copy has landed
                // and every MMA that read it has completed once this
                // accumulator is ready), so the fp32 partial goes there, row
                // by row with 16-byte units XOR-swizzled by row (conflict-free
                // stores by the row-owning lanes).  An empty k-range
                // contributes zeros.
                constexpr uint32_t ROW_BYTES = (uint32_t)BN * 4;
                static_assert((uint32_t)AROWS * ROW_BYTES <= (uint32_t)STAGES * Cf::STAGE_BYTES,
                              "partial tile fits the ring");
                const int kc = p.s.kc;
                const int part = (int)cluster_ctarank();  // = u.slot: CTA c is part c mod kc
                const bool empty = u.k1 <= u.k0;
                fence_proxy_async_smem();
                const uint32_t srow = sbase + (uint32_t)row_in_tile * ROW_BYTES;
#pragma unroll 1
                for (int j = 0; j < BN / 32; ++j) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(tbase + j * 32, r);
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const int unit = (j * 8 + v) ^ (row_in_tile & 7);
                            st_shared_u4(srow + (uint32_t)(unit * 16), empty ? 0u : r[4 * v],
                                         empty ? 0u : r[4 * v + 1], empty ? 0u : r[4 * v + 2],
                                         empty ? 0u : r[4 * v + 3]);
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(buf));
                // Every row of this part is in shared memory.  The barrier
                // orders all epilogue threads' stores before thread 0's
                // release-arrives on the other CTAs' barriers; their acquire
                // waits then see the whole partial.
                // (The test hook skips this CTA's signals, so the other parts'
                // waits run out: they record a timeout and store nothing.)
                named_bar_sync(BAR_EPI_SYNC, EPI_THREADS);
                if (et == 0 && cta != p.inject_skip_cta) {
#pragma unroll 1
                    for (int q2 = 0; q2 < kc; ++q2)
                        if (q2 != part) mbar_arrive_cluster(mapa_shared(parts_bar, (uint32_t)q2));
                }
                const bool got = mbar_wait_acq_cluster(parts_bar, 0, p.wait_limit_ns);
                if (!epi_vote_all(got)) {
                    if (et == 0) record_status(p.status, STATUS_FLAG_TIMEOUT);
                } else {
                    uint8_t* ctile = reinterpret_cast<uint8_t*>(p.C) + (size_t)tm * BM * p.ldc * 2;
                    const int col0 = u.tn * BN;
                    if (kc == 2)
                        cluster_reduce_slice<2, BN, OUT_BF16>(sbase, part, rows_valid, et, ctile, p.ldc, col0, p.N);
                    else if (kc == 4)
                        cluster_reduce_slice<4, BN, OUT_BF16>(sbase, part, rows_valid, et, ctile, p.ldc, col0, p.N);
                    else
                        cluster_reduce_slice<8, BN, OUT_BF16>(sbase, part, rows_valid, et, ctile, p.ldc, col0, p.N);
                }
            } else {
            if (u.role == ROLE_PEER) {
                // fp32 partial -> this CTA's slot, laid out [chunk][vec][row] so
                // a warp's 16-byte stores cover 512 contiguous bytes
                float4* slot =
                    reinterpret_cast<float4*>(p.partials + (size_t)(u.slot * CM + rank) * BM * BN);
#pragma unroll 1
                for (int j = 0; j < BN / 32; ++j) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(tbase + j * 32, r);
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            st_f4(slot + (size_t)(j * 8 + v) * BM + row_in_tile,
                                  make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                              __uint_as_float(r[4 * v + 2]),
                                              __uint_as_float(r[4 * v + 3])));
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR_MMA)
                        mbar_arrive_cluster(mapa_shared(tempty_bar(buf), 0));
                    else
                        mbar_arrive(tempty_bar(buf));
                }
                // The barrier orders every epilogue thread's partial stores
                // before thread 0's post, and the post is a release at GPU
                // scope: an owner that acquires the flag sees all of them.
                named_bar_sync(BAR_EPI_SYNC, EPI_THREADS);
                if (et == 0 && cta != p.inject_skip_cta) post_flag(p.flags + u.tile * CM + rank, p.epoch);
            } else {
                bool store = true;
                if (u.role == ROLE_OWNER) {
                    const uint64_t target = ((uint64_t)p.epoch << 32) | (uint32_t)u.npeers;
                    // one thread polls (128 pollers per owner slowed the L2);
                    // the vote is the barrier that orders the other threads'
                    // reads of the partials after its acquire
                    const bool got = et != 0 || wait_flag(p.flags + u.tile * CM + rank, target, p.wait_limit_ns);
                    store = epi_vote_all(got);
                    if (!store && et == 0) record_status(p.status, STATUS_FLAG_TIMEOUT);
                }
                // The CTA's last unit: every load into the ring has landed and
                // every MMA that read it has completed (this accumulator is
                // ready), so the ring is idle and the epilogue may use it:
                //  * C: the converted tile is staged in the ring and written
                //    out row by row (a warp's store covers 512 contiguous
                //    bytes instead of 16 bytes in each of 32 rows);
                //  * OWNER: the first `staged` peers' partials of all chunks
                //    are copied in at once, one round trip to L2 instead of one
                //    per chunk; the additions keep the ascending k order.
                // Ring layout: [C: SROWS rows x BN halves, 16-byte units
                // XOR-swizzled by row][partials: chunk][peer][vec][row] float4.
                Cursor peek = cur;
                Unit next_unit;
                const bool last = !cursor_next(p.s, unit_cta, peek, next_unit);
                constexpr int SROWS = AROWS;  // rows a CTA can hold valid
                constexpr int C_UNITS = BN / 8;  // 16-byte units in a staged row
                constexpr uint32_t C_STAGE_BYTES = (uint32_t)SROWS * BN * 2;
                constexpr uint32_t PEER_STAGE_BYTES = (uint32_t)BN * SROWS * 4;
                constexpr uint32_t RING_BYTES = (uint32_t)STAGES * Cf::STAGE_BYTES;
                static_assert(C_STAGE_BYTES <= RING_BYTES, "C tile fits the ring");
                // All peers beside the C tile when they fit; else all peers with C
                // stored straight from registers; else as many as fit beside C.
                bool c_staged = last;
                int staged = 0;
                if (last && u.role == ROLE_OWNER && store) {
                    const uint32_t all_peers = (uint32_t)u.npeers * PEER_STAGE_BYTES;
                    if (C_STAGE_BYTES + all_peers > RING_BYTES && all_peers <= RING_BYTES)
                        c_staged = false;
                    staged = c_staged
                                 ? min(u.npeers, (int)((RING_BYTES - C_STAGE_BYTES) / PEER_STAGE_BYTES))
                                 : u.npeers;
                }
                const uint32_t pstage = sbase + (c_staged ? C_STAGE_BYTES : 0u);
                if (last) fence_proxy_async_smem();  // the ring was last used by the async proxy
                if (staged > 0) {
                    if (row_ok && staged > 0) {
                        const float4* part = reinterpret_cast<const float4*>(p.partials);
                        const size_t slot_f4 = (size_t)BM * BN / 4;
#pragma unroll 1
                        for (int j = 0; j < BN / 32; ++j) {
#pragma unroll 1
                            for (int q = 0; q < staged; ++q) {
                                const float4* src = part + (size_t)((u.slot + q) * CM + rank) * slot_f4 +
                                                    (size_t)(j * 8) * BM + row_in_tile;
                                const uint32_t dst =
                                    pstage + (uint32_t)((((j * staged + q) * 8) * SROWS + row_in_tile) * 16);
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    cp_async_16(dst + (uint32_t)(v * SROWS * 16), src + (size_t)v * BM);
                            }
                        }
                        cp_async_wait_all();
                    }
                }
                uint8_t* crow = reinterpret_cast<uint8_t*>(p.C) + ((size_t)row * p.ldc) * 2;
                // pair MMA, a tile in mid-stream (its ring is busy): C through
                // tensor copies when the plan has a tensor map for C
                const bool c_box = Cf::EPI_STAGE_BYTES > 0 && p.c_tma && store && !c_staged;
#pragma unroll 1
                for (int j = 0; j < BN / 32; ++j) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld_32x32b_x32(tbase + j * 32, r);
                    float acc[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(r[i]);
                    if (u.role == ROLE_OWNER && store && row_ok) {
                        // staged peers first (the lowest k), from shared memory
#pragma unroll 1
                        for (int q = 0; q < staged; ++q) {
                            const uint32_t sp =
                                pstage + (uint32_t)((((j * staged + q) * 8) * SROWS + row_in_tile) * 16);
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                const float4 x = ld_shared_f4(sp + (uint32_t)(v * SROWS * 16));
                                acc[4 * v] += x.x;
                                acc[4 * v + 1] += x.y;
                                acc[4 * v + 2] += x.z;
                                acc[4 * v + 3] += x.w;
                            }
                        }
                        // peers in ascending k: slots u.slot, u.slot + 1, ... (this half)
                        // Loads of PEER_BATCH peers are issued before any of them is
                        // added, so 32 16-byte loads per thread are in flight; the
                        // additions keep the ascending order.
                        constexpr int PEER_BATCH = 4;
                        const float4* base = reinterpret_cast<const float4*>(p.partials) +
                                             (size_t)(j * 8) * BM + row_in_tile;
                        const size_t slot_f4 = (size_t)BM * BN / 4;
#pragma unroll 1
                        for (int pp = staged + 1; pp <= u.npeers; pp += PEER_BATCH) {
                            float4 x[PEER_BATCH][8];
#pragma unroll
                            for (int q = 0; q < PEER_BATCH; ++q) {
                                if (pp + q <= u.npeers) {
                                    const float4* slot =
                                        base + (size_t)((u.slot + pp - 1 + q) * CM + rank) * slot_f4;
#pragma unroll
                                    for (int v = 0; v < 8; ++v) x[q][v] = ld_cg_f4(slot + (size_t)v * BM);
                                }
                            }
#pragma unroll
                            for (int q = 0; q < PEER_BATCH; ++q) {
                                if (pp + q <= u.npeers) {
#pragma unroll
                                    for (int v = 0; v < 8; ++v) {
                                        acc[4 * v] += x[q][v].x;
                                        acc[4 * v + 1] += x[q][v].y;
                                        acc[4 * v + 2] += x[q][v].z;
                                        acc[4 * v + 3] += x[q][v].w;
                                    }
                                }
                            }
                        }
                    }
                    if (c_box) {
                        // Two 32-column chunks make one 64-column box of the warp's
                        // 32 rows.  It is staged in the warp's own 4 KB, 16-byte units
                        // XOR-swizzled by row (the layout of a 128-byte-swizzled
                        // tensor box; conflict-free writes by the row-owning lanes),
                        // and written by one tensor copy: full 128-byte lines to L2
                        // instead of 16 bytes in each of 32 rows per store.
                        const uint32_t stg = epi_stage + (uint32_t)((warp & 3) * 4096);
                        if ((j & 1) == 0) {
                            // the previous box's copy has read the buffer
                            if (lane == 0) bulk_wait_group_read_0();
                            __syncwarp();
                        }
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int unit = ((j & 1) * 4 + v) ^ (lane & 7);
                            st_shared_u4(stg + (uint32_t)(lane * 128 + unit * 16),
                                         pack2<OUT_BF16>(acc[8 * v], acc[8 * v + 1]),
                                         pack2<OUT_BF16>(acc[8 * v + 2], acc[8 * v + 3]),
                                         pack2<OUT_BF16>(acc[8 * v + 4], acc[8 * v + 5]),
                                         pack2<OUT_BF16>(acc[8 * v + 6], acc[8 * v + 7]));
                        }
                        if (j & 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int x = u.tn * BN + (j - 1) * 32;  // multiple of 64
                                const int y = tm * BM + (warp & 3) * 32;
                                if (x < p.N && y < p.M) tma_store_2d(&tmC, stg, x, y);
                                bulk_commit_group();
                            }
                        }
                    } else if (store && row_ok) {
                        if (c_staged) {
                            const uint32_t srow = sbase + (uint32_t)(row_in_tile * BN * 2);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const int unit = (j * 4 + v) ^ (row_in_tile & (C_UNITS - 1));
                                st_shared_u4(srow + (uint32_t)(unit * 16),
                                             pack2<OUT_BF16>(acc[8 * v], acc[8 * v + 1]),
                                             pack2<OUT_BF16>(acc[8 * v + 2], acc[8 * v + 3]),
                                             pack2<OUT_BF16>(acc[8 * v + 4], acc[8 * v + 5]),
                                             pack2<OUT_BF16>(acc[8 * v + 6], acc[8 * v + 7]));
                            }
                        } else {
                            const int col0 = u.tn * BN + j * 32;
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const int col = col0 + 8 * v;
                                if (col < p.N)
                                    st_u4(crow + (size_t)col * 2, pack2<OUT_BF16>(acc[8 * v], acc[8 * v + 1]),
                                          pack2<OUT_BF16>(acc[8 * v + 2], acc[8 * v + 3]),
                                          pack2<OUT_BF16>(acc[8 * v + 4], acc[8 * v + 5]),
                                          pack2<OUT_BF16>(acc[8 * v + 6], acc[8 * v + 7]));
                            }
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR_MMA)
                        mbar_arrive_cluster(mapa_shared(tempty_bar(buf), 0));
                    else
                        mbar_arrive(tempty_bar(buf));
                }
                if (c_staged && store) {
                    // every epilogue warp has staged its rows; write whole rows:
                    // lane l takes unit l % C_UNITS of row i * (32 / C_UNITS) + l / C_UNITS
                    named_bar_sync(BAR_EPI_SYNC, EPI_THREADS);
                    constexpr int ROWS_PER_STORE = 32 / C_UNITS;
                    const int unit = lane % C_UNITS;
                    const int col = u.tn * BN + unit * 8;
                    const int first = (et >> 5) * ROWS_PER_STORE + lane / C_UNITS;
#pragma unroll 4
                    for (int r = first; r < rows_valid; r += 4 * ROWS_PER_STORE) {
                        const uint4 v = ld_shared_u4(sbase + (uint32_t)(r * BN * 2) +
                                                     (uint32_t)((unit ^ (r & (C_UNITS - 1))) * 16));
                        if (col < p.N)
                            st_u4(reinterpret_cast<uint8_t*>(p.C) + ((size_t)(tm * BM + r) * p.ldc + col) * 2,
                                  v.x, v.y, v.z, v.w);
                    }
                }
            }
            }  // not a cluster split-K part
            ++iter;
        }
        // every tensor copy of C has completed before the CTA ends
        if (Cf::EPI_STAGE_BYTES > 0 && p.c_tma && lane == 0) bulk_wait_group_0();
    }

    tc_fence_before_sync();
    __syncwarp();
    if constexpr (CM == 2 || KCL) {
        // no CTA leaves while another may still signal it or read its
        // shared memory
        cluster_sync_all();
    } else {
        __syncthreads();
    }
    if (p.trace && threadIdx.x == 0) {
        p.trace[(size_t)cta * TRACE_N + TRACE_END] = globaltimer_ns();
        p.trace[(size_t)cta * TRACE_N + TRACE_CLK_END] = sm_clock64();
        p.trace[(size_t)cta * TRACE_N + TRACE_CLK_START] = c_start;
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        if constexpr (PAIR_MMA)
            tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cf::TMEM_COLS);
    }
}

}  // namespace psm
