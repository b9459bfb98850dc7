"""Pins of the oracle's index / ancestor-mask construction.

The oracle finds ancestor sets by walking parent links; these tests check
them against the recurrence anc[t] = anc[parent[t]] | {t} and against
subtree membership found by a depth-first search over child lists, for
every tree with T <= 6. The combined key list is pinned by a closed form
(contiguous placement gives 0..n-1) and by slot-multiset equality.
"""

import itertools

import numpy as np
import pytest

import oracle
from workloads import make_config, make_inputs


def _all_trees(T):
    for choice in itertools.product(*[range(i) for i in range(1, T)]):
        yield [-1] + list(choice)


def _subtree_members(par, T):
    children = [[] for _ in range(T)]
    for i in range(1, T):
        children[par[i]].append(i)
    sub = []
    for u in range(T):
        seen, stack = set(), [u]
        while stack:
            x = stack.pop()
            seen.add(x)
            stack.extend(children[x])
        sub.append(seen)
    return sub


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6])
def test_ancestor_masks_exhaustive(T):
    for par in _all_trees(T):
        inp = make_inputs(batch=1, num_heads=1, prefix=[2], T=T, tree=par, pool_slots=64,
                          nsplit=1, seed=1)
        _, _, anc = oracle.build_meta(inp)
        anc = [int(x) for x in anc[0]]
        # Recurrence form.
        rec = [0] * T
        for t in range(T):
            rec[t] = (rec[par[t]] if par[t] >= 0 else 0) | (1 << t)
        assert anc == rec
        # u is an ancestor-or-self of t  <=>  t lies in u's subtree.
        sub = _subtree_members(par, T)
        for t in range(T):
            for u in range(T):
                assert bool((anc[t] >> u) & 1) == (t in sub[u])
        # popcount = depth + 1, and bit t is always set.
        for t in range(T):
            d, v = 0, par[t]
            while v != -1:
                d, v = d + 1, par[v]
            assert bin(anc[t]).count("1") == d + 1
            assert (anc[t] >> t) & 1


def test_chain_and_star_closed_forms():
    T = 64
    inp = make_inputs(batch=1, num_heads=1, prefix=[1], T=T, tree="chain", pool_slots=256,
                      nsplit=1, seed=2)
    _, _, anc = oracle.build_meta(inp)
    assert [int(x) for x in anc[0]] == [(1 << (t + 1)) - 1 if t < 63 else (1 << 64) - 1
                                        for t in range(T)]
    inp = make_inputs(batch=1, num_heads=1, prefix=[1], T=T, tree="star", pool_slots=256,
                      nsplit=1, seed=2)
    _, _, anc = oracle.build_meta(inp)
    assert [int(x) for x in anc[0]] == [1] + [1 | (1 << t) for t in range(1, T)]


@pytest.mark.parametrize("B,L", [(1, [0]), (2, [5, 0]), (8, [3, 1, 4, 1, 5, 9, 2, 6])])
def test_indices_contiguous_closed_form(B, L):
    """Contiguous placement assigns slots in logical order, so the combined list
    is exactly 0..n-1 and the offsets are the running sums of L_b + T."""
    T = 3
    inp = make_inputs(batch=B, num_heads=1, prefix=L, T=T, tree="random", pool_slots=512,
                      nsplit=2, seed=3, placement="contiguous")
    indptr, indices, _ = oracle.build_meta(inp)
    n = sum(L) + B * T
    assert np.array_equal(indices, np.arange(n, dtype=np.int32))
    assert indptr.tolist() == [0] + list(np.cumsum([x + T for x in L]))


def test_indices_scattered_is_a_relabelling():
    """Scattered placement: same per-request lengths, and the list is the
    contiguous one relabelled through the slot map (a permutation of used
    slots), so the two lists are equal as multisets of distinct slots."""
    a = make_inputs(batch=3, num_heads=1, prefix=[7, 0, 11], T=5, tree="random",
                    pool_slots=4096, nsplit=2, seed=4, placement="scattered")
    ipa, ixa, anca = oracle.build_meta(a)
    c = make_inputs(batch=3, num_heads=1, prefix=[7, 0, 11], T=5, tree="random",
                    pool_slots=4096, nsplit=2, seed=4, placement="contiguous")
    ipc, ixc, ancc = oracle.build_meta(c)
    assert np.array_equal(ipa, ipc) and np.array_equal(anca, ancc)
    assert len(set(ixa.tolist())) == len(ixa) == len(ixc)
    # The content at each logical position is the same row of values.
    assert np.array_equal(a.kv_pool[ixa], c.kv_pool[ixc])


def test_config_sizes():
    for idx, n_expected in [(1, 260), (2, 4112)]:
        inp = make_config(idx)
        indptr, indices, anc = oracle.build_meta(inp)
        assert indptr[-1] == n_expected == len(indices)
        assert anc.shape == (inp.batch, inp.T)
