// Tile scheduler: one definition used by the device kernel and by the host
// plan (which enumerates the same units for inspection and tests).
//
// Work decomposition (GitHub issue "Stream-k matmul implementation very slow
// mostly because of if/else inside for loop", final code version):
//  * the wrapper's tile grid, iterations per tile, Stream-K tile count
//    (tiles mod g, plus g with the "two_tiles" rule) and the even split of
//    the Stream-K iterations, the first `rem` CTAs taking one more;
//  * first_wave: a CTA's iteration range cut at tile boundaries into units;
//  * full_tiles: whole tiles numbered after the Stream-K tiles;
//  * swizzle_tile / linear_tile: the raster (grouped by GROUP_M rows, or
//    row-major).
// A third raster follows a Hilbert curve (the blog summary "Inside NVIDIA
// GPUs: Anatomy of high performance matmul kernels" lists Hilbert-curve
// scheduling among the Hopper tricks): the plan builds the order on the
// host, and tile_coords reads it from a table.
// The persistent schedule (HF post "naive vs persistent matmul") is the same
// machinery with no Stream-K tiles and a grid of one CTA per SM; the
// data-parallel schedule launches one CTA per tile.
//
// Split-K (GitHub issue above, closing comments: a fixed split of K as the
// alternative decomposition): every tile's k-range is cut into `split`
// near-equal parts; units are numbered part-major with the k = 0 parts (the
// owners) last, and a persistent grid takes units c, c + grid, ...  A CTA
// therefore finishes all its peer units before any owner unit, and owners
// wait only on peers, which never wait.
//
// Cluster split-K (the same fixed split, reduced on chip): CTA c computes
// part c mod kc of tile c / kc, once; the kc CTAs of a tile form one
// thread-block cluster and add their fp32 partials through distributed
// shared memory in ascending part order, so no workspace is involved.
//
// Fixup roles.  A unit that starts at k-iteration 0 of its tile and ends
// before the tile's last iteration is the OWNER; a unit that starts past
// iteration 0 is a PEER.  A CTA's range is contiguous, so only its first unit
// can be a PEER and only its last can be an OWNER.  The peers of an owner in
// CTA c are CTAs c+1 .. c+npeers, in ascending k.  Every unit carries the
// partial-tile slot it writes (PEER) or the first slot it reads (OWNER); an
// owner's peers occupy consecutive slots in ascending k.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define PSM_HD __host__ __device__ __forceinline__
#else
#define PSM_HD inline
#endif

namespace psm {

enum : int32_t { ROLE_FULL = 0, ROLE_OWNER = 1, ROLE_PEER = 2, ROLE_CLUSTER_PART = 3 };

struct Sched {
    int32_t tiles_m, tiles_n, tiles;
    int32_t ipt;         // k-iterations per tile
    int32_t group_m;     // rows of tiles per raster group, 0 = linear raster
    int32_t grid;        // CTAs launched
    int32_t sk_tiles;    // raster ids [0, sk_tiles) are split by Stream-K
    int32_t persistent;  // 1: CTA c takes whole tiles sk+c, sk+c+grid, ...
    int32_t split;       // split-K parts per tile (0: no split-K)
    int32_t k_rotate;    // 1: whole tiles start their k loop at their own
                         // offset (see unit_kblock)
    int32_t l2_prefetch; // k-blocks of B to prefetch into L2 ahead of the ring (0: off)
    int32_t kc;          // cluster split-K: parts per tile = CTAs per cluster (0: off)
    const int32_t* raster_table;  // optional: tile id -> (row << 16) | column
    int64_t sk_q;        // Stream-K iterations per CTA (floor)
    int64_t sk_r;        // CTAs [0, sk_r) take sk_q + 1
};

struct Unit {
    int32_t tile;    // raster id
    int32_t k0, k1;  // k-iterations [k0, k1)
    int32_t role;
    int32_t npeers;  // OWNER: peers it adds; CLUSTER_PART: the other parts of its tile
    int32_t tm, tn;  // tile row / column
    int32_t slot;    // PEER: its partial-tile slot; OWNER: slot of its first
                     // peer (the peers' slots follow in ascending k);
                     // CLUSTER_PART: its part (= its rank in the cluster)
};

struct Cursor {
    int64_t it, it_end;   // remaining Stream-K iterations of this CTA
    int32_t next_whole;   // next whole tile, >= tiles when done
};

PSM_HD int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// k-block visited at step i of a unit.  Partial units walk [k0, k1) in order.
// With k_rotate, a whole tile t starts at block floor(t * ipt / tiles) and
// wraps around: when one row of tiles streams a B that is read exactly once,
// the tiles then read different rows of B at any moment instead of all
// crowding the same few, which spreads the reads over the DRAM channels.
// Only the fp32 summation order of such a tile changes.
PSM_HD int32_t unit_kblock(const Sched& s, int32_t tile, int32_t k0, int32_t k1, int32_t i) {
    if (s.k_rotate && k0 == 0 && k1 == s.ipt) {
        const int32_t rot = (int32_t)(((int64_t)tile * s.ipt) / (s.tiles > 0 ? s.tiles : 1));
        const int32_t kb = i + rot;
        return kb >= s.ipt ? kb - s.ipt : kb;
    }
    return k0 + i;
}

PSM_HD void tile_coords(const Sched& s, int32_t t, int32_t& tm, int32_t& tn) {
    if (s.raster_table) {
        const int32_t v = s.raster_table[t];
        tm = v >> 16;
        tn = v & 0xFFFF;
    } else if (s.group_m > 0) {
        int32_t width = s.group_m * s.tiles_n;
        int32_t gid = t / width;
        int32_t first = gid * s.group_m;
        int32_t gsize = s.tiles_m - first < s.group_m ? s.tiles_m - first : s.group_m;
        tm = first + (t % gsize);
        tn = (t % width) / gsize;
    } else {
        tm = t / s.tiles_n;
        tn = t % s.tiles_n;
    }
}

// first Stream-K iteration of CTA c
PSM_HD int64_t sk_begin(const Sched& s, int64_t c) {
    return c * s.sk_q + imin64(c, s.sk_r);
}

// CTA whose Stream-K range holds global iteration `it`
PSM_HD int64_t sk_cta_of(const Sched& s, int64_t it) {
    int64_t big = s.sk_r * (s.sk_q + 1);  // iterations held by the CTAs with one extra
    if (it < big) return it / (s.sk_q + 1);
    return s.sk_r + (it - big) / s.sk_q;  // sk_q > 0 here: otherwise big == total
}

PSM_HD void cursor_init(const Sched& s, int32_t cta, Cursor& c) {
    if (s.sk_tiles > 0) {
        c.it = sk_begin(s, cta);
        c.it_end = sk_begin(s, (int64_t)cta + 1);
    } else {
        c.it = c.it_end = 0;
    }
    c.next_whole = s.sk_tiles + cta;  // split-K: the unit counter
}

PSM_HD bool cursor_next(const Sched& s, int32_t cta, Cursor& c, Unit& u) {
    if (c.it < c.it_end) {
        int64_t tile = c.it / s.ipt;
        int64_t tile_first = tile * s.ipt;
        int64_t k0 = c.it - tile_first;
        int64_t end = imin64(tile_first + s.ipt, c.it_end);
        u.tile = (int32_t)tile;
        u.k0 = (int32_t)k0;
        u.k1 = (int32_t)(end - tile_first);
        c.it = end;
        u.slot = cta;
        if (u.k0 > 0) {
            u.role = ROLE_PEER;
            u.npeers = 0;
        } else if (u.k1 == s.ipt) {
            u.role = ROLE_FULL;
            u.npeers = 0;
        } else {
            u.role = ROLE_OWNER;
            u.npeers = (int32_t)(sk_cta_of(s, tile_first + s.ipt - 1) - cta);
            u.slot = cta + 1;
        }
        tile_coords(s, u.tile, u.tm, u.tn);
        return true;
    }
    if (s.kc > 0) {
        const int64_t total = (int64_t)s.tiles * s.kc;
        if (c.next_whole >= total) return false;
        const int64_t uid = c.next_whole;
        c.next_whole = 0x7FFFFFFF;  // one unit per CTA
        const int32_t part = (int32_t)(uid % s.kc);
        u.tile = (int32_t)(uid / s.kc);
        u.k0 = (int32_t)(((int64_t)part * s.ipt) / s.kc);
        u.k1 = (int32_t)(((int64_t)(part + 1) * s.ipt) / s.kc);
        u.role = ROLE_CLUSTER_PART;
        u.npeers = s.kc - 1;
        u.slot = part;
        tile_coords(s, u.tile, u.tm, u.tn);
        return true;
    }
    if (s.split > 0) {
        const int64_t total = (int64_t)s.tiles * s.split;
        if (c.next_whole >= total) return false;
        const int64_t uid = c.next_whole;
        c.next_whole += s.grid;
        const int32_t part = s.split - 1 - (int32_t)(uid / s.tiles);
        u.tile = (int32_t)(uid % s.tiles);
        u.k0 = (int32_t)(((int64_t)part * s.ipt) / s.split);
        u.k1 = (int32_t)(((int64_t)(part + 1) * s.ipt) / s.split);
        const int32_t first_peer_slot = u.tile * (s.split - 1);
        if (s.split == 1) {
            u.role = ROLE_FULL;
            u.npeers = 0;
            u.slot = 0;
        } else if (part == 0) {
            u.role = ROLE_OWNER;
            u.npeers = s.split - 1;
            u.slot = first_peer_slot;
        } else {
            u.role = ROLE_PEER;
            u.npeers = 0;
            u.slot = first_peer_slot + part - 1;
        }
        tile_coords(s, u.tile, u.tm, u.tn);
        return true;
    }
    if (c.next_whole < s.tiles) {
        u.tile = c.next_whole;
        u.k0 = 0;
        u.k1 = s.ipt;
        u.role = ROLE_FULL;
        u.npeers = 0;
        u.slot = 0;
        tile_coords(s, u.tile, u.tm, u.tn);
        c.next_whole = s.persistent ? c.next_whole + s.grid : s.tiles;
        return true;
    }
    return false;
}

}  // namespace psm
