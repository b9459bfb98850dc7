"""The KV partition rules of the split-KV kernels (csrc/partition.h), compiled
on the CPU with g++ and checked against what the method needs of them: the
nsplit partitions of a request's keys tile [0, K) in order, cut at key-tile
boundaries; the tensor-core kernels' wave-shaped split keeps every partition
non-empty once there are 2 * nsplit tiles, gives the items of the last,
partial wave of resident clusters one tile each, and shares the rest evenly;
and the first index of the partial wave is the largest multiple of the
resident count (or the item count when there is at most one wave). The
two-SM kernel's one-wave split cuts the keys, not tiles, evenly over as
many partitions as one wave of resident clusters holds."""

import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mla_speculative_decoding_gb300", "csrc")

HARNESS = r'''
#include <cstdio>
#include "partition.h"
using namespace mlav;
int main() {
    const int tile = 256;
    const int Ks[] = {0, 1, 255, 256, 257, 4096, 4112, 32768, 65552, 184792, 200000};
    const int nsplits[] = {1, 4, 8, 64, 128};
    const int nrbs[] = {1, 2, 4};
    const int batches[] = {1, 3, 8};
    const int residents[] = {0, 36, 76, 1000};
    for (int K : Ks) for (int ns : nsplits) for (int nrb : nrbs) for (int B : batches)
    for (int res : residents) {
        const long long items = (long long)B * ns * nrb;
        const int full = wave_full_items(items, res);
        printf("W %lld %d %d\n", items, res, full);
        for (int b = 0; b < B; ++b) for (int rb = 0; rb < nrb; ++rb) {
            const int item0 = b * nrb + rb;  // partition-major dispatch
            for (int s = 0; s < ns; ++s) {
                int beg, end;
                split_range_waves(K, ns, s, tile, item0, B * nrb, full, beg, end);
                printf("P %d %d %d %d %d %d %d %d %d %d\n", K, ns, nrb, B, res, b, rb, s, beg, end);
            }
        }
    }
    for (int K : Ks) for (int ns : nsplits) for (int s = 0; s < ns; ++s) {
        int beg, end;
        split_range_tiles(K, ns, s, tile, beg, end);
        printf("T %d %d %d %d %d\n", K, ns, s, beg, end);
    }
    for (int K : Ks) for (int ns : nsplits) for (int s = 0; s < ns + 2; ++s) {
        int beg, end;
        split_range_keys(K, ns, s, beg, end);
        printf("K %d %d %d %d %d\n", K, ns, s, beg, end);
    }
    for (int K : Ks) for (int ns : nsplits) for (int s = 0; s < ns + 2; ++s) {
        int beg, end;
        split_range_one_wave(K, ns, s, tile, beg, end);
        printf("Q %d %d %d %d %d\n", K, ns, s, beg, end);
    }
    const long long pairs[] = {0, 1, 2, 16, 19, 76, 77, 1000};
    const int res2[] = {-1, 0, 36, 76};
    for (long long p : pairs) for (int r : res2) for (int ns : nsplits)
        printf("O %lld %d %d %d\n", p, r, ns, one_wave_parts(p, r, ns));
    return 0;
}
'''


@pytest.fixture(scope="module")
def harness_out(tmp_path_factory):
    d = tmp_path_factory.mktemp("partition")
    src, exe = d / "harness.cpp", d / "harness"
    src.write_text(HARNESS)
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout


@pytest.fixture(scope="module")
def key_table(harness_out):
    keys, owp, onew = {}, [], {}
    for line in harness_out.splitlines():
        f = line.split()
        if f[0] == "K":
            K, ns, s, beg, end = (int(x) for x in f[1:])
            keys.setdefault((K, ns), []).append((s, beg, end))
        elif f[0] == "Q":
            K, ns, s, beg, end = (int(x) for x in f[1:])
            onew.setdefault((K, ns), []).append((s, beg, end))
        elif f[0] == "O":
            owp.append(tuple(int(x) for x in f[1:]))
    return keys, owp, onew


@pytest.fixture(scope="module")
def table(harness_out):
    waves, parts, even = [], {}, {}
    for line in harness_out.splitlines():
        f = line.split()
        if f[0] in ("K", "O", "Q"):
            continue
        if f[0] == "W":
            waves.append(tuple(int(x) for x in f[1:]))
        elif f[0] == "P":
            K, ns, nrb, B, res, b, rb, s, beg, end = (int(x) for x in f[1:])
            parts.setdefault((K, ns, nrb, B, res, b, rb), []).append((s, beg, end))
        else:
            K, ns, s, beg, end = (int(x) for x in f[1:])
            even.setdefault((K, ns), []).append((s, beg, end))
    return waves, parts, even


def _check_cover(K, ranges, tile=256):
    pos = 0
    for _, beg, end in ranges:
        assert beg == pos and end >= beg, (K, ranges)
        assert (beg % tile == 0 or beg == K) and (end % tile == 0 or end == K)
        pos = end
    assert pos == K


def test_wave_boundary(table):
    waves, _, _ = table
    for items, res, full in waves:
        if res <= 0 or items <= res:
            assert full == items
        else:
            assert full % res == 0 and full <= items < full + res


def test_even_tile_split_covers_and_balances(table):
    _, _, even = table
    for (K, ns), ranges in even.items():
        _check_cover(K, ranges)
        tiles = [-(-(e - b) // 256) for _, b, e in ranges]
        assert max(tiles) - min(tiles) <= 1 and tiles == sorted(tiles, reverse=True)


def test_wave_shaped_split(table):
    waves, parts, _ = table
    full_of = {(items, res): full for items, res, full in waves}
    n_tail_cases = 0
    for (K, ns, nrb, B, res, b, rb), ranges in parts.items():
        _check_cover(K, ranges)
        tiles = -(-K // 256)
        full = full_of[(B * ns * nrb, res)]
        item = [(s * B + b) * nrb + rb for s, _, _ in ranges]
        tail = [i >= full for i in item]
        sizes = [-(-(e - beg) // 256) for _, beg, e in ranges]
        if tiles >= 2 * ns:
            assert min(sizes) >= 1, "every partition keeps a tile"
        if any(tail) and not all(tail) and tiles >= 2 * ns:
            n_tail_cases += 1
            assert all(sz == 1 for sz, t in zip(sizes, tail) if t)
            head = [sz for sz, t in zip(sizes, tail) if not t]
            assert max(head) - min(head) <= 1 and head == sorted(head, reverse=True)
            assert all(t2 >= t1 for t1, t2 in zip(tail, tail[1:])), "the tail is a suffix"
        else:
            assert max(sizes) - min(sizes) <= 1
    assert n_tail_cases > 0


def test_long_workload_shape(table):
    """184,792 keys, 64 partitions, 2 row blocks, 36 resident four-SM clusters:
    partitions 54-63 take one tile each, the first 54 share the other 712."""
    _, parts, _ = table
    for rb in (0, 1):
        ranges = parts[(184792, 64, 2, 1, 36, 0, rb)]
        sizes = [-(-(e - b) // 256) for _, b, e in ranges]
        assert sizes[54:] == [1] * 10
        assert sum(sizes[:54]) == 722 - 10 and set(sizes[:54]) <= {13, 14}


PLAN_HARNESS = r'''
#include <cstdio>
#include <vector>
#include <random>
#include "partition.h"
using namespace mlav;
int main() {
    std::mt19937 rng(7);
    const int Cs[] = {1, 5, 36, 76};
    for (int trial = 0; trial < 400; ++trial) {
        const int B = 1 + rng() % 12, nrb = 1 + rng() % 5, nsplit = 1 + rng() % 64;
        std::vector<int> t(B), ptile(B + 1, 0);
        for (int b = 0; b < B; ++b) {
            const int r = rng() % 10;
            t[b] = r == 0 ? 0 : (r < 4 ? 1 + rng() % 3 : 1 + rng() % 900);
            ptile[b + 1] = ptile[b] + t[b] * nrb;
        }
        int tmax = 0;
        for (int x : t) tmax = x > tmax ? x : tmax;
        const int w = ptile[B];
        for (int C : Cs) {
            const bool fits = plan_fits(w, tmax, C, nsplit);
            printf("F %d %d %d %d %d %d %d\n", trial, C, w, nrb, nsplit, tmax, fits ? 1 : 0);
            for (int b = 0; b < B; ++b) printf("T %d %d %d %d\n", trial, C, b, t[b]);
            if (!fits) continue;
            for (int c = 0; c < C; ++c) {
                int x = plan_begin(c, C, w);
                const int xend = plan_begin(c + 1, C, w);
                printf("R %d %d %d %d %d\n", trial, C, c, x, xend);
                int b = 0;
                while (x < xend) {
                    int rb, u0, u1, s;
                    const int n = plan_step(ptile.data(), nrb, C, w, c, x, xend, b, rb, u0, u1, s);
                    printf("I %d %d %d %d %d %d %d %d\n", trial, C, c, b, rb, u0, u1, s);
                    if (n <= 0) return 1;
                    x += n;
                }
            }
            for (int b = 0; b < B; ++b)
                for (int rb = 0; rb < nrb; ++rb) {
                    const int s0 = ptile[b] + rb * t[b];
                    printf("O %d %d %d %d %d %d\n", trial, C, b, rb, plan_pair_owner(s0, t[b], C, w),
                           plan_pair_parts(s0, t[b], C, w));
                }
        }
    }
    return 0;
}
'''


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    d = tmp_path_factory.mktemp("plan")
    src, exe = d / "plan.cpp", d / "plan"
    src.write_text(PLAN_HARNESS)
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    cases = {}
    for line in out.splitlines():
        f = line.split()
        key = (int(f[1]), int(f[2]))
        c = cases.setdefault(key, {"t": {}, "ranges": {}, "items": [], "owners": {}})
        v = [int(x) for x in f[3:]]
        if f[0] == "F":
            c["w"], c["nrb"], c["nsplit"], c["tmax"], c["fits"] = v
        elif f[0] == "T":
            c["t"][v[0]] = v[1]
        elif f[0] == "R":
            c["ranges"][v[0]] = (v[1], v[2])
        elif f[0] == "I":
            c["items"].append(tuple(v))
        else:
            c["owners"][(v[0], v[1])] = (v[2], v[3])
    return cases


def test_balanced_plan(plan):
    """Every (request, row block) pair's tiles are covered once, in key
    order, by partitions 0, 1, 2, ... (fewer than nsplit) held by clusters
    in increasing order (consecutive ones when every cluster holds a tile);
    cluster loads differ by at most one tile; each pair
    has one owner cluster, which holds its first tile, and its part count
    equals the partitions the walk produced."""
    n_fit = 0
    for (trial, C), c in plan.items():
        if not c["fits"]:
            # refused only when some pair could be cut into more than nsplit parts
            m = c["w"] // C
            bound = c["tmax"] if m == 0 else (c["tmax"] - 1 + m - 1) // m + 1
            assert c["w"] == 0 or bound > c["nsplit"]
            continue
        n_fit += 1
        w, nrb = c["w"], c["nrb"]
        sizes = [e - b for b, e in (c["ranges"][k] for k in range(C))]
        assert sum(sizes) == w and max(sizes) - min(sizes) <= 1
        pos = {}
        for cl, b, rb, u0, u1, s in c["items"]:
            assert 0 <= s < c["nsplit"] and u1 > u0
            cov = pos.setdefault((b, rb), [])
            cov.append((u0, u1, s, cl))
        for b, t in c["t"].items():
            for rb in range(nrb):
                cov = sorted(pos.get((b, rb), []))
                if t == 0:
                    assert not cov
                else:
                    assert cov[0][0] == 0 and cov[-1][1] == t
                    assert all(x[1] == y[0] for x, y in zip(cov, cov[1:]))
                    assert [x[2] for x in cov] == list(range(len(cov)))
                    assert all(y[3] > x[3] for x, y in zip(cov, cov[1:]))
                    if w >= C:  # every cluster holds a tile: the holders are consecutive
                        assert all(y[3] == x[3] + 1 for x, y in zip(cov, cov[1:]))
                owner, parts = c["owners"][(b, rb)]
                assert 0 <= owner < C and parts == len(cov)
                if cov:
                    assert owner == cov[0][3]
    assert n_fit > 100


def test_long_workload_plan():
    """The long workload (184,792 keys: 722 tiles per row block, 2 row
    blocks) on 36 clusters: one item of 40-41 tiles per cluster, 18
    partitions per row block."""
    ptile, C = [0, 2 * 722], 36
    w = ptile[-1]
    sizes = [0] * C
    parts = {0: 0, 1: 0}
    exe_free = [(c, (c * w) // C, ((c + 1) * w) // C) for c in range(C)]
    for c, b0, e0 in exe_free:
        sizes[c] = e0 - b0
        parts[b0 // 722] += 1
        assert b0 // 722 == (e0 - 1) // 722, "no cluster spans both row blocks"
    assert set(sizes) <= {40, 41} and parts == {0: 18, 1: 18}


def test_even_key_split(key_table):
    """split_range_keys: partitions 0..parts-1 tile [0, K) in order with sizes
    that differ by at most one key, the largest one ceil(K / parts) keys in
    no more 256-key tiles than the largest tile-aligned partition; those at
    or past `parts` are empty at K. The mid workload (65,552 keys over 64
    partitions) gets 16 partitions of 1025 keys and 48 of 1024."""
    keys, _, _ = key_table
    for (K, ns), ranges in keys.items():
        ranges.sort()
        pos = 0
        for s, beg, end in ranges:
            if s >= ns:
                assert beg == end == K
                continue
            assert beg == pos and end >= beg
            pos = end
        assert pos == K
        sizes = [e - b for s, b, e in ranges if s < ns]
        assert max(sizes) - min(sizes) <= 1 and max(sizes) == -(-K // ns)
        tiles = -(-K // 256)
        assert -(-max(sizes) // 256) == -(-tiles // ns)
    mid = [e - b for s, b, e in sorted(keys[(65552, 64)]) if s < 64]
    assert sorted(mid) == [1024] * 48 + [1025] * 16


def test_one_wave_parts(key_table):
    """Partitions per pair for the one-wave split: floor(resident / pairs)
    capped at nsplit, and 0 (the wave-shaped split) when the pairs exceed one
    wave or the resident count is unknown."""
    _, owp, _ = key_table
    for pairs, res, ns, got in owp:
        if res <= 0 or pairs <= 0 or pairs > res:
            assert got == 0
        else:
            assert got == min(ns, res // pairs) and got >= 1
    got = {(p, r, n): g for p, r, n, g in owp}
    assert got[(1, 76, 64)] == 64      # the mid workload: all 64 partitions in one wave
    assert got[(16, 76, 8)] == 4       # sparse decode: 16 requests x 4 partitions
    assert got[(77, 76, 64)] == 0      # more pairs than clusters: wave-shaped


def test_one_wave_split(key_table):
    """split_range_one_wave: with no more tiles than partitions, the even key
    split; otherwise tile-aligned ranges in order whose tile counts differ by
    at most one, the larger ones last (so the last, partly filled tile sits
    in one of them); partitions at or past `parts` are empty. The mid
    workload (65,552 keys = 256 full tiles and one of 16 keys, 64
    partitions): partitions 0-62 take 4 full tiles, partition 63 four and
    the 16-key one."""
    keys, _, onew = key_table
    for (K, ns), ranges in onew.items():
        ranges.sort()
        tiles = -(-K // 256)
        if tiles <= ns:
            assert ranges == sorted(keys[(K, ns)])
            continue
        pos, sizes = 0, []
        for s, beg, end in ranges:
            if s >= ns:
                assert beg == end == K
                continue
            assert beg == pos and end > beg
            assert beg % 256 == 0 and (end % 256 == 0 or end == K)
            sizes.append(-(-(end - beg) // 256))
            pos = end
        assert pos == K
        assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes)
    mid = sorted(onew[(65552, 64)])
    assert all(e - b == 1024 for s, b, e in mid[:63])
    assert (mid[63][1], mid[63][2]) == (64512, 65552)
