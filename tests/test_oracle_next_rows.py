"""Pins for the oracle of the steps beside the verify attention (greedy tree
acceptance, KV relocation, fp8 paged indexer logits): closed forms, an
independent property check, a library special case (torch's float8 type and
fp64 matmul) and the placement invariance of the attention itself."""

import numpy as np
import pytest
import torch

import oracle
from workloads import (make_accept_inputs, make_indexer_inputs, make_inputs,
                       make_relocate_inputs)


# ---------------------------------------------------------------- tree acceptance
def _check_acceptance(par, tok, tgt, loc, commit, an, ks, nt):
    """Independent statement of greedy acceptance as properties of the result."""
    T = len(par)
    n = int(commit) - 1
    path = [0] + [int(x) for x in an[:n]]
    assert all(x == -1 for x in an[n:])
    for a, c in zip(path[:-1], path[1:]):
        assert par[c] == a, "consecutive path nodes are parent and child"
        assert tok[c] == tgt[a], "each accepted node's token is the target's choice"
        # the lowest-numbered matching child is taken
        first = min(k for k in range(1, T) if par[k] == a and tok[k] == tgt[a])
        assert c == first
    last = path[-1]
    assert not any(par[k] == last and tok[k] == tgt[last] for k in range(1, T)), "maximal"
    assert list(nt[:n + 1]) == [int(tok[c]) for c in path[1:]] + [int(tgt[last])]
    assert all(x == -1 for x in nt[n + 1:])
    assert list(ks[:n + 1]) == [int(loc[c]) for c in path]
    assert all(x == -1 for x in ks[n + 1:])


def test_accept_chain_all_match():
    T = 9
    par = np.array([[-1] + list(range(T - 1))], np.int32)
    tok = np.arange(100, 100 + T, dtype=np.int32)[None]
    tgt = np.array([[100 + t + 1 for t in range(T)]], np.int32)  # node t predicts node t+1's token
    loc = np.arange(7, 7 + T, dtype=np.int32)[None]
    c, an, ks, nt = oracle.tree_accept(par, tok, tgt, loc)
    assert c[0] == T
    assert list(an[0][:T - 1]) == list(range(1, T))
    assert list(ks[0]) == list(range(7, 7 + T))
    assert list(nt[0]) == list(range(101, 100 + T)) + [100 + T]


def test_accept_nothing_matches():
    par = np.array([[-1, 0, 0, 1]], np.int32)
    tok = np.array([[5, 6, 7, 8]], np.int32)
    tgt = np.array([[9, 9, 9, 9]], np.int32)
    loc = np.array([[40, 41, 42, 43]], np.int32)
    c, an, ks, nt = oracle.tree_accept(par, tok, tgt, loc)
    assert c[0] == 1 and nt[0][0] == 9 and ks[0][0] == 40
    assert (an[0] == -1).all() and (nt[0][1:] == -1).all() and (ks[0][1:] == -1).all()


def test_accept_repeated_sibling_token_takes_lowest_node():
    par = np.array([[-1, 0, 0, 0, 2, 1]], np.int32)
    tok = np.array([[0, 4, 4, 3, 6, 6]], np.int32)
    tgt = np.array([[4, 6, 6, 0, 0, 0]], np.int32)
    loc = np.arange(6, dtype=np.int32)[None]
    c, an, ks, nt = oracle.tree_accept(par, tok, tgt, loc)
    assert list(an[0][:2]) == [1, 5] and c[0] == 3 and list(nt[0][:3]) == [4, 6, 0]


@pytest.mark.parametrize("tree", ["random", "chain", "star"])
@pytest.mark.parametrize("match", [0.0, 0.5, 0.9, 1.0])
def test_accept_properties_random(tree, match):
    for seed in range(6):
        x = make_accept_inputs(batch=5, T=24, tree=tree, vocab=7, match=match, seed=seed)
        c, an, ks, nt = oracle.tree_accept(x.tree_parent, x.draft_tokens, x.target_argmax,
                                           x.out_cache_loc)
        for b in range(5):
            _check_acceptance(x.tree_parent[b], x.draft_tokens[b], x.target_argmax[b],
                              x.out_cache_loc[b], c[b], an[b], ks[b], nt[b])


def test_accept_rejects_bad_tree():
    par = np.array([[-1, 0, 3, 1]], np.int32)
    z = np.zeros((1, 4), np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.tree_accept(par, z, z, z)


# ---------------------------------------------------------------- KV relocation
def _relocatable_verify(batch=3, seed=3):
    """A verify workload on contiguous slots 0..n-1 of a pool with a free top
    part, plus contiguous free destination ranges for every request's prefix."""
    L = [900, 0, 333][:batch]
    inp = make_inputs(batch=batch, num_heads=4, prefix=L, T=8, tree="random", pool_slots=8192,
                      nsplit=4, seed=seed, placement="contiguous")
    n = sum(L) + batch * 8
    dst = (n + 5 + np.concatenate([[0], np.cumsum(L)[:-1]])).astype(np.int32)
    return inp, dst


def test_relocation_keeps_attention_bitwise():
    """Moving a request's prefix rows changes where they live, not what they
    hold: the oracle's attention over the relocated state is bit-identical
    (a relocation that dropped, duplicated or reordered a row would not be)."""
    inp, dst = _relocatable_verify()
    ip, ix, _ = oracle.build_meta(inp)
    ref_out, ref_lse = oracle.verify_attention(inp, ip, ix)
    pool, r2t, prog = oracle.kv_relocate(inp.kv_pool, inp.req_to_token, inp.req_pool_indices,
                                         inp.prefix_lens, dst, np.zeros(3, np.int32), 10_000)
    assert list(prog) == list(inp.prefix_lens)
    inp.kv_pool, inp.req_to_token = pool, r2t
    ip2, ix2, _ = oracle.build_meta(inp)
    out, lse = oracle.verify_attention(inp, ip2, ix2)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)
    for b in range(3):
        row = r2t[inp.req_pool_indices[b]]
        L = inp.prefix_lens[b]
        assert list(row[:L]) == list(range(dst[b], dst[b] + L))


def test_relocation_budget_progress_and_exact_copies():
    x = make_relocate_inputs(batch=4, prefix=[70, 5, 0, 130], pool_slots=1024, seed=7)
    pool, r2t, prog = x.kv_pool, x.req_to_token, x.progress
    budget = 32
    calls = 0
    while (prog < x.prefix_lens).any():
        before_prog = prog.copy()
        new_pool, new_r2t, new_prog = oracle.kv_relocate(pool, r2t, x.req_pool_indices,
                                                         x.prefix_lens, x.dst_start, prog, budget)
        assert list(new_prog) == [min(int(l), int(p) + budget) for l, p in zip(x.prefix_lens, before_prog)]
        for b in range(4):
            row_old, row_new = r2t[x.req_pool_indices[b]], new_r2t[x.req_pool_indices[b]]
            for j in range(int(before_prog[b]), int(new_prog[b])):
                assert row_new[j] == x.dst_start[b] + j
                assert np.array_equal(new_pool[row_new[j]], pool[row_old[j]])
            assert np.array_equal(row_new[new_prog[b]:], row_old[new_prog[b]:])
        changed = np.nonzero((new_pool != pool).any(axis=1))[0]
        moved = {int(x.dst_start[b] + j) for b in range(4)
                 for j in range(int(before_prog[b]), int(new_prog[b]))}
        assert set(changed.tolist()) <= moved
        pool, r2t, prog = new_pool, new_r2t, new_prog
        calls += 1
    assert calls == 5  # ceil(130 / 32)


def test_relocation_in_place_rows_and_contract():
    x = make_relocate_inputs(batch=2, prefix=[40, 20], pool_slots=256, seed=9, in_place=10)
    pool, r2t, prog = oracle.kv_relocate(x.kv_pool, x.req_to_token, x.req_pool_indices,
                                         x.prefix_lens, x.dst_start, x.progress, 1000)
    assert list(prog) == [40, 20]
    # a destination range that covers a live source slot is refused
    bad = x.dst_start.copy()
    bad[1] = int(x.req_to_token[x.req_pool_indices[0], 15])
    with pytest.raises(oracle.OracleError):
        oracle.kv_relocate(x.kv_pool, x.req_to_token, x.req_pool_indices, x.prefix_lens, bad,
                           x.progress, 1000)


# ---------------------------------------------------------------- fp8 indexer
def test_e4m3_decoding_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def _torch_indexer(ix):
    """The indexer written with torch fp64 ops: decode, matmul, relu, weighted
    head sum, scale; -inf past each request's length."""
    q = torch.from_numpy(ix.q).view(torch.float8_e4m3fn).to(torch.float64)
    B, H, _ = q.shape
    P = ix.block_table.shape[1]
    out = torch.full((B, P * 64), float("-inf"), dtype=torch.float64)
    kv = torch.from_numpy(ix.kv_blocks)
    w = torch.from_numpy(ix.weights).to(torch.float64)
    for b in range(B):
        for p in range(P):
            n = min(64, int(ix.seq_lens[b]) - 64 * p)
            if n <= 0:
                continue
            blk = kv[int(ix.block_table[b, p])]
            k = blk[:8192].view(torch.float8_e4m3fn).reshape(64, 128).to(torch.float64)
            sc = blk[8192:].view(torch.float32).to(torch.float64)
            logit = (torch.relu(q[b] @ k.T) * w[b][:, None]).sum(0) * sc
            out[b, 64 * p:64 * p + n] = logit[:n]
    return out.numpy()


@pytest.mark.parametrize("lens", [[1, 64, 65, 200], [0, 129, 3, 640]])
def test_indexer_matches_torch_fp64(lens):
    ix = make_indexer_inputs(batch=4, num_heads=16, seq_lens=lens, max_pages=11, seed=sum(lens))
    got = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table, ix.seq_lens)
    ref = _torch_indexer(ix)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.allclose(got[fin], ref[fin], rtol=1e-12, atol=1e-12)
    for b, l in enumerate(lens):
        assert np.isneginf(got[b, l:]).all() and np.isfinite(got[b, :l]).all()


def test_indexer_page_table_indirection_invariance():
    ix = make_indexer_inputs(batch=3, num_heads=8, seq_lens=[300, 70, 128], max_pages=5, seed=5)
    base = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table, ix.seq_lens)
    perm = np.random.default_rng(0).permutation(ix.kv_blocks.shape[0])
    inv = np.argsort(perm)
    kv2 = ix.kv_blocks[perm]                     # block perm[i] now lives at i
    bt2 = np.where(ix.block_table >= 0, inv[np.maximum(ix.block_table, 0)], -1).astype(np.int32)
    moved = oracle.fp8_indexer_logits(ix.q, ix.weights, kv2, bt2, ix.seq_lens)
    assert np.array_equal(base, moved)


def test_indexer_zero_query_and_relu():
    ix = make_indexer_inputs(batch=2, num_heads=4, seq_lens=[100, 10], max_pages=2, seed=6)
    zero = oracle.fp8_indexer_logits(np.zeros_like(ix.q), ix.weights, ix.kv_blocks,
                                     ix.block_table, ix.seq_lens)
    assert (zero[0, :100] == 0).all() and (zero[1, :10] == 0).all()
    # a head whose query is the negation of a key scores that key 0 (ReLU)
    q = np.zeros_like(ix.q)
    blk = ix.kv_blocks[ix.block_table[0, 0]]
    q[0, 0] = blk[:128] ^ 0x80                   # sign flipped: dot = -|k|^2 < 0
    w = np.ones_like(ix.weights)
    out = oracle.fp8_indexer_logits(q, w, ix.kv_blocks, ix.block_table, ix.seq_lens)
    assert out[0, 0] == 0.0
