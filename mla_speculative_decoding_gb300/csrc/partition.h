// Partitions of a request's keys over the split-KV work items. Plain C++
// (no CUDA headers): shared by the kernels and by the host, and compiled on
// its own by the CPU test of the partition rules.
#pragma once

#ifdef __CUDACC__
#define MLAV_HD __host__ __device__
#else
#define MLAV_HD
#endif

namespace mlav {

MLAV_HD inline int mlav_min(int a, int b) { return a < b ? a : b; }

// Key range of split s of a request with K keys: contiguous ranges of
// ceil(K / nsplit) keys; trailing splits may be empty.
MLAV_HD inline void split_range(int K, int nsplit, int s, int& beg, int& end) {
    const int chunk = (K + nsplit - 1) / nsplit;
    beg = mlav_min(K, s * chunk);
    end = mlav_min(K, beg + chunk);
}

// Tile-aligned variant for kernels that walk the keys in tiles of `tile`:
// the ceil(K / tile) tiles are spread as evenly as possible (the first
// tiles % nsplit splits take one more), so no split carries a mostly empty
// last tile and the longer work items come first in launch order.
MLAV_HD inline void split_range_tiles(int K, int nsplit, int s, int tile, int& beg, int& end) {
    const int tiles = (K + tile - 1) / tile;
    const int base = tiles / nsplit, rem = tiles % nsplit;
    const int t0 = s * base + mlav_min(s, rem);
    const int nt = base + (s < rem ? 1 : 0);
    beg = mlav_min(K, t0 * tile);
    end = mlav_min(K, (t0 + nt) * tile);
}

// Wave-shaped variant for launches whose work items run in waves of resident
// clusters, dispatched in index order: the item of partition s is item0 +
// s * stride. Items at or past index `full` (the items of the last, partial
// wave) get one tile each, and the partitions before them share the
// remaining tiles evenly as in split_range_tiles, so that the full waves end
// together and the partial wave is as short as possible. Every partition
// keeps at least one tile. Falls back to split_range_tiles when nothing is
// in the partial wave, when the whole range is, or when there are fewer than
// 2 * nsplit tiles.
MLAV_HD inline void split_range_waves(int K, int nsplit, int s, int tile, int item0, int stride,
                                      int full, int& beg, int& end) {
    const int tiles = (K + tile - 1) / tile;
    const int last = item0 + (nsplit - 1) * stride;  // item of the last partition
    const int s_tail = last < full ? nsplit : (full <= item0 ? 0 : (full - item0 + stride - 1) / stride);
    const int n_tail = nsplit - s_tail;
    if (n_tail == 0 || s_tail == 0 || tiles < 2 * nsplit) {
        split_range_tiles(K, nsplit, s, tile, beg, end);
        return;
    }
    const int head = tiles - n_tail;  // tiles of partitions [0, s_tail)
    int t0, nt;
    if (s < s_tail) {
        const int base = head / s_tail, rem = head % s_tail;
        t0 = s * base + mlav_min(s, rem);
        nt = base + (s < rem ? 1 : 0);
    } else {
        t0 = head + (s - s_tail);
        nt = 1;
    }
    beg = mlav_min(K, t0 * tile);
    end = mlav_min(K, (t0 + nt) * tile);
}

// Even split of K keys over `parts` partitions for launches in which all of
// them run at once: partition s < parts takes keys [floor(s K / parts),
// floor((s + 1) K / parts)), so sizes differ by at most one key and a
// request's largest partition holds ceil(K / parts) keys (the same number of
// 256-key tiles as the largest tile-aligned partition, but no more keys);
// partitions at or past `parts` are empty.
MLAV_HD inline void split_range_keys(int K, int parts, int s, int& beg, int& end) {
    if (parts <= 0 || s >= parts) {
        beg = end = K;
        return;
    }
    beg = (int)((long long)K * s / parts);
    end = (int)((long long)K * (s + 1) / parts);
}

// Split of K keys over `parts` partitions that all run at once (one wave):
// with no more tiles than partitions, the even key split (every partition at
// most one tile, as few keys as possible); otherwise whole tiles, shared as
// evenly as possible with the extra tiles on the last partitions, so that
// the request's last, partly filled tile is one of them and as few
// partitions as possible hold a tile more than the rest.
MLAV_HD inline void split_range_one_wave(int K, int parts, int s, int tile, int& beg, int& end) {
    const int tiles = (K + tile - 1) / tile;
    if (tiles <= parts || s >= parts) {
        split_range_keys(K, parts, s, beg, end);
        return;
    }
    const int base = tiles / parts, lo = parts - tiles % parts;  // partitions [lo, parts) take base + 1
    const int t0 = s * base + (s > lo ? s - lo : 0);
    const int nt = base + (s >= lo ? 1 : 0);
    beg = mlav_min(K, t0 * tile);
    end = mlav_min(K, (t0 + nt) * tile);
}

// Partitions per (request, row block) pair for a launch of `pairs` pairs on
// `resident` clusters of one CTA pair each when each partition is one
// cluster: as many as one wave of resident clusters holds, at most nsplit;
// 0 (no even key split: the wave-shaped split instead) when the pairs do not
// fit one wave or the resident count is unknown.
inline int one_wave_parts(long long pairs, int resident, int nsplit) {
    if (resident <= 0 || pairs <= 0 || pairs > resident) return 0;
    const long long p = resident / pairs;
    return (int)(p < nsplit ? p : nsplit);
}

// Index of the first item of the last, partial wave when `items` work items
// run on `resident` clusters at a time (items when every wave is full or
// when there is no more than one wave, or the resident count is unknown).
inline int wave_full_items(long long items, int resident) {
    if (resident <= 0 || items <= resident) return (int)items;
    return (int)((items / resident) * resident);
}

// Balanced plan for persistent clusters. The key tiles of every (request,
// row block) pair, request major and row block minor, form one sequence of
// w tiles; request b's pairs start at ptile[b] (ptile[batch] = w) and hold
// (ptile[b + 1] - ptile[b]) / nrb tiles each. Cluster c of C takes tiles
// [plan_begin(c), plan_begin(c + 1)); the part of a pair one cluster holds
// is one partition of that pair's rows, numbered in key order from 0.
MLAV_HD inline int plan_begin(int c, int C, int w) { return (int)((long long)c * w / C); }

// The cluster holding tile x (0 <= x < w).
MLAV_HD inline int plan_cluster(int x, int C, int w) { return (int)(((long long)(x + 1) * C - 1) / w); }

// Whether no pair of at most tmax tiles is cut into more than nsplit parts:
// clusters hold at least floor(w / C) tiles, so a pair of t tiles meets at
// most ceil((t - 1) / floor(w / C)) + 1 of them (t of them when a cluster
// may hold no tile at all).
MLAV_HD inline bool plan_fits(long long w, int tmax, int C, int nsplit) {
    if (w <= 0 || w > (1ll << 30) || C <= 0) return false;
    const long long m = w / C;
    const long long parts = m == 0 ? tmax : (tmax - 1 + m - 1) / m + 1;
    return parts <= nsplit;
}

// Partition of the pair starting at tile s0 that holds its tile x: the
// clusters met since s0 (every cluster holds a tile when w >= C; otherwise
// each holds at most one, and the count is the tile offset).
MLAV_HD inline int plan_part(int s0, int x, int C, int w) {
    return w >= C ? plan_cluster(x, C, w) - plan_cluster(s0, C, w) : x - s0;
}

// Parts of the pair whose t tiles start at tile s0, and the cluster that
// writes its empty partitions (the one holding its first tile; for a pair
// without tiles, the one holding the tile at its place, or the last).
MLAV_HD inline int plan_pair_parts(int s0, int t, int C, int w) {
    return t > 0 ? plan_part(s0, s0 + t - 1, C, w) + 1 : 0;
}
MLAV_HD inline int plan_pair_owner(int s0, int t, int C, int w) {
    return plan_cluster(t > 0 ? s0 : (s0 < w - 1 ? s0 : w - 1), C, w);
}

// One step of cluster `cid`'s walk from its tile x (< xend): the pair
// holding x is request b (advanced past requests that end at or before x)
// and row block rb; the step takes that pair's tiles [u0, u1), partition s.
// Returns the number of tiles taken.
MLAV_HD inline int plan_step(const int* ptile, int nrb, int C, int w, int cid, int x, int xend, int& b,
                             int& rb, int& u0, int& u1, int& s) {
    while (ptile[b + 1] <= x) ++b;
    const int p0 = ptile[b];
    const int t = (ptile[b + 1] - p0) / nrb;
    const int off = x - p0;
    rb = off / t;
    u0 = off - rb * t;
    u1 = mlav_min(t, u0 + (xend - x));
    s = plan_part(p0 + rb * t, x, C, w);
    (void)cid;
    return u1 - u0;
}

}  // namespace mlav
