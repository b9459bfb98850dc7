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

// Index of the first item of the last, partial wave when `items` work items
// run on `resident` clusters at a time (items when every wave is full or
// when there is no more than one wave, or the resident count is unknown).
inline int wave_full_items(long long items, int resident) {
    if (resident <= 0 || items <= resident) return (int)items;
    return (int)((items / resident) * resident);
}

}  // namespace mlav
