// schedule.h -- the persistent tile schedule of the tensor-core GEMM kernel,
// shared by the kernel (device) and the host planner, and compiled on its own
// by a CPU test that checks it.
//
// G clusters (CTA pairs) run the kernel; each owns a list of work units.
//   * Whole tiles: tiles 0 .. first-1, where first = tiles - tail_tiles, are
//     dealt round robin (cluster c takes c, c + G, c + 2G, ...), every K
//     block of a tile in one unit.
//   * Stream-K tail: the tail_tiles * num_kb K blocks of the last tail_tiles
//     tiles (tile-major, K blocks in order) are cut into tail_clusters
//     consecutive ranges of nearly equal length; cluster c < tail_clusters
//     takes range c, one unit per tile the range touches.  When
//     tail_clusters is a multiple s of tail_tiles, every range lies inside
//     one tile (each tail tile in s parts, one per cluster).
// A range may start inside a tile, so a tile's K blocks can be spread over
// several consecutive clusters c0 < c1 < ... .  The unit holding the tile's
// first K block (cluster c0) owns the tile: it adds, in K order, the FP32
// sums that clusters c0+1 .. c0+others leave in their slots, and writes C.
// Only a range's first unit can start inside a tile, so a cluster leaves sums
// in at most one slot (its own index), and an owning unit that is split is
// the last unit of its range: the clusters it waits for publish their first
// unit and never wait themselves, so no wait can close a cycle.
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define EMU_HD __host__ __device__ __forceinline__
#else
#define EMU_HD inline
#endif

namespace emu {

struct TileSchedule {
    int tiles;           // tiles_m * tiles_n
    int num_kb;          // K blocks per tile
    int tail_tiles;      // tiles in the stream-K tail (0: none)
    int tail_clusters;   // clusters sharing the tail (0 when tail_tiles is 0)
    int clusters;        // G: clusters the kernel runs
};

struct Unit {
    int tile, kb0, kb1;  // K blocks [kb0, kb1) of `tile`
    int publish;         // >= 0: a later part of the tile: leave the sums in this slot
    int others;          // owner: the slots of clusters c+1 .. c+others follow, in K order
};

// First K block (tail-relative) of cluster c's range.
EMU_HD int64_t sk_range_start(const TileSchedule& s, int c) {
    const int64_t W = static_cast<int64_t>(s.tail_tiles) * s.num_kb;
    return static_cast<int64_t>(c) * W / s.tail_clusters;
}

// Cluster whose range holds tail K block x: the largest c with
// sk_range_start(c) <= x, i.e. floor(((x + 1) * Ct - 1) / W).
EMU_HD int sk_cluster_of(const TileSchedule& s, int64_t x) {
    const int64_t W = static_cast<int64_t>(s.tail_tiles) * s.num_kb;
    return static_cast<int>(((x + 1) * s.tail_clusters - 1) / W);
}

EMU_HD int sched_whole_units(const TileSchedule& s, int c) {
    const int first = s.tiles - s.tail_tiles;
    return c < first ? (first - c + s.clusters - 1) / s.clusters : 0;
}

// Number of units of cluster c.
EMU_HD int sched_units(const TileSchedule& s, int c) {
    int n = sched_whole_units(s, c);
    if (s.tail_tiles > 0 && c < s.tail_clusters) {
        const int64_t a = sk_range_start(s, c), b = sk_range_start(s, c + 1);
        if (b > a) n += static_cast<int>((b - 1) / s.num_kb - a / s.num_kb + 1);
    }
    return n;
}

// Unit i (0 <= i < sched_units(s, c)) of cluster c.
EMU_HD Unit sched_unit(const TileSchedule& s, int c, int i) {
    Unit w;
    const int whole = sched_whole_units(s, c);
    if (i < whole) {
        w.tile = c + i * s.clusters;
        w.kb0 = 0;
        w.kb1 = s.num_kb;
        w.publish = -1;
        w.others = 0;
        return w;
    }
    const int64_t a = sk_range_start(s, c), b = sk_range_start(s, c + 1);
    const int64_t t = a / s.num_kb + (i - whole);            // tail tile index
    const int64_t t0 = t * s.num_kb;                           // its first tail K block
    const int64_t lo = a > t0 ? a : t0;
    const int64_t hi = b < t0 + s.num_kb ? b : t0 + s.num_kb;
    w.tile = s.tiles - s.tail_tiles + static_cast<int>(t);
    w.kb0 = static_cast<int>(lo - t0);
    w.kb1 = static_cast<int>(hi - t0);
    if (w.kb0 > 0) {
        w.publish = c;
        w.others = 0;
    } else {
        w.publish = -1;
        w.others = sk_cluster_of(s, t0 + s.num_kb - 1) - c;
    }
    return w;
}

// The tail of a GEMM of `tiles` tiles of num_kb K blocks on `resident`
// clusters.  None when the tiles fill whole rounds.  Otherwise the r =
// tiles % resident tiles of the last round are shared by Ct clusters, the
// cheapest plan by a cost in half K blocks.  Handing one part's sums to the
// owner (one FP32 slot written, then read) costs fix2 half blocks (it
// depends on how long a K block of the mode takes; measured with up to 8
// parts per tile).  An owner reads its parts one after another, so each
// part past the 8th adds rd = (fix2 + 2) / 3 half blocks (reading a slot is
// about a third of the hand-over: 1.5 of 5.5 us for a 256-wide tile).
//   * aligned: Ct = s r, 2 <= s <= min(resident / r, num_kb / 2): every
//     range lies inside one tile, each cluster makes one hand-over:
//     cost 2 ceil(num_kb / s) + fix2 + max(s - 8, 0) rd;
//   * stream-K: 2 <= Ct <= min(resident, r num_kb / 2): ranges of two K
//     blocks or more that may cross tiles, so a cluster can both publish
//     (its first part) and own (its last), and a tile has up to ceil(Ct / r)
//     parts: cost 2 ceil(W / Ct) + 2 fix2 + max(ceil(Ct / r) - 8, 0) rd,
//     W = r num_kb.
// Every s and Ct is tried, the larger first (a tie keeps the wider split;
// up to 8 parts a tile the costs fall as s and Ct grow).  The tail is split
// only when the cheapest cost beats the unsplit round (2 num_kb) by at least
// a whole K block.  A few deep tiles (a weight gradient: 256 x 256 with K in
// the millions) are then spread over every resident cluster.
EMU_HD void sched_plan_tail(int tiles, int num_kb, int resident, int fix2, int* tail_tiles,
                            int* tail_clusters) {
    *tail_tiles = 0;
    *tail_clusters = 0;
    if (resident <= 0 || num_kb < 2) return;
    const int r = tiles % resident;
    if (r == 0) return;
    const int64_t W = static_cast<int64_t>(r) * num_kb;
    const int64_t rd = (fix2 + 2) / 3;
    int64_t best = 2 * static_cast<int64_t>(num_kb) - 1;    // a cost must be below this
    int64_t best_ct = 0;
    int smax = resident / r;
    if (smax > num_kb / 2) smax = num_kb / 2;
    for (int s = smax; s >= 2; --s) {
        const int64_t cost = 2 * ((num_kb + s - 1) / s) + fix2 + (s > 8 ? s - 8 : 0) * rd;
        if (cost < best) {
            best = cost;
            best_ct = static_cast<int64_t>(s) * r;
        }
    }
    int64_t cmax = resident;
    if (cmax > W / 2) cmax = W / 2;
    for (int64_t ct = cmax; ct >= 2; --ct) {
        if (ct % r == 0 && ct / r <= smax) continue;        // the aligned plan above
        const int64_t parts = (ct + r - 1) / r;
        const int64_t cost = 2 * ((W + ct - 1) / ct) + 2 * static_cast<int64_t>(fix2) +
                             (parts > 8 ? parts - 8 : 0) * rd;
        if (cost < best) {
            best = cost;
            best_ct = ct;
        }
    }
    if (best_ct == 0) return;
    *tail_tiles = r;
    *tail_clusters = static_cast<int>(best_ct);
}

// Clusters the kernel runs: whole rounds of `resident` when there are whole
// tiles before a tail (the round robin's stride must be the clusters the tail
// was planned for), the tail's clusters when the tail is all there is, and
// otherwise one cluster per tile up to `resident`.
EMU_HD int sched_grid_clusters(int tiles, int tail_tiles, int tail_clusters, int resident) {
    if (tail_tiles == 0) return tiles < resident ? tiles : resident;
    return tiles > tail_tiles ? resident : tail_clusters;
}

}  // namespace emu
