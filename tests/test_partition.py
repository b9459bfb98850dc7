"""The KV partition rules of the split-KV kernels (csrc/partition.h), compiled
on the CPU with g++ and checked against what the method needs of them: the
nsplit partitions of a request's keys tile [0, K) in order, cut at key-tile
boundaries; the tensor-core kernels' wave-shaped split keeps every partition
non-empty once there are 2 * nsplit tiles, gives the items of the last,
partial wave of resident clusters one tile each, and shares the rest evenly;
and the first index of the partial wave is the largest multiple of the
resident count (or the item count when there is at most one wave)."""

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
    return 0;
}
'''


@pytest.fixture(scope="module")
def table(tmp_path_factory):
    d = tmp_path_factory.mktemp("partition")
    src, exe = d / "harness.cpp", d / "harness"
    src.write_text(HARNESS)
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    waves, parts, even = [], {}, {}
    for line in out.splitlines():
        f = line.split()
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
