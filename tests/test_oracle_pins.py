"""Pins of the CPU oracle's attention to things other than itself.

Each test fixes the oracle against brute force, a library special case, a
closed form or an invariant, so that a plausible slip (a dropped prefix,
missing self-visibility, the wrong V dims, a wrong scale or log base, a
transposed tree index) fails at least one of them.
"""

import itertools

import numpy as np
import pytest
import torch

import oracle
from tests.brute import brute_row, visible_slots
from workloads import bf16_bits_to_f32, make_config, make_inputs


def _oracle(inp, rows=None):
    ip, ix, _ = oracle.build_meta(inp)
    return oracle.verify_attention(inp, ip, ix, rows=rows)


@pytest.mark.parametrize("seed,B,H,L,T,tree", [
    (11, 1, 1, [3], 1, "chain"),
    (12, 1, 2, [8], 4, "random"),
    (13, 2, 2, [5, 0], 4, "random"),
    (14, 2, 1, [0, 7], 3, "star"),
    (15, 2, 2, [8, 2], 4, [-1, 0, 0, 2]),
])
def test_brute_force_tiny(seed, B, H, L, T, tree):
    """Whole definition on tiny inputs: oracle == pure-Python brute force."""
    inp = make_inputs(batch=B, num_heads=H, prefix=L, T=T, tree=tree, pool_slots=64,
                      nsplit=2, seed=seed)
    out, lse = _oracle(inp)
    for n in range(inp.num_rows):
        bo, bl = brute_row(inp, n)
        np.testing.assert_allclose(out[n], bo, rtol=0, atol=1e-12)
        assert abs(lse[n] - bl) <= 1e-12


def _sdpa_chain_case(B, H, L, T, seed):
    inp = make_inputs(batch=B, num_heads=H, prefix=[L] * B, T=T, tree="chain", pool_slots=4096,
                      nsplit=4, seed=seed)
    out, _ = _oracle(inp)
    out = out.reshape(B, T, H, 512)
    for b in range(B):
        # Keys in logical order for the last token (whose visible set is all
        # L + T keys of a chain).
        slots = visible_slots(inp, b, T - 1)
        kv = torch.from_numpy(bf16_bits_to_f32(inp.kv_pool[slots]).astype(np.float64))
        q = torch.from_numpy(bf16_bits_to_f32(inp.q[b * T:(b + 1) * T]).astype(np.float64))
        qh = q.permute(1, 0, 2).unsqueeze(0)                      # [1, H, T, 576]
        k = kv.unsqueeze(0).unsqueeze(0).expand(1, H, L + T, 576)
        v = kv[:, :512].unsqueeze(0).unsqueeze(0).expand(1, H, L + T, 512)
        mask = torch.ones(T, L + T, dtype=torch.bool)
        mask[:, L:] = torch.tril(torch.ones(T, T, dtype=torch.bool))
        ref = torch.nn.functional.scaled_dot_product_attention(
            qh, k, v, attn_mask=mask, scale=inp.softmax_scale)      # [1, H, T, 512]
        got = torch.from_numpy(out[b]).permute(1, 0, 2)            # [H, T, 512]
        torch.testing.assert_close(got, ref[0], rtol=0, atol=1e-12)


def test_chain_tree_is_causal_attention():
    """A chain tree (parent i-1) is causal attention over prefix + tree: equals
    torch's fp64 scaled_dot_product_attention with a prefix-open, lower-
    triangular mask (and the single latent row broadcast to all heads)."""
    _sdpa_chain_case(B=2, H=3, L=37, T=6, seed=21)


def test_chain_no_prefix_is_is_causal():
    """L = 0 chain: plain causal self-attention (is_causal=True), no explicit mask."""
    T, H = 9, 2
    inp = make_inputs(batch=1, num_heads=H, prefix=[0], T=T, tree="chain", pool_slots=256,
                      nsplit=1, seed=22)
    out, _ = _oracle(inp)
    kv = torch.from_numpy(bf16_bits_to_f32(inp.kv_pool[inp.out_cache_loc]).astype(np.float64))
    q = torch.from_numpy(bf16_bits_to_f32(inp.q).astype(np.float64)).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, kv[None, None].expand(1, H, T, 576), kv[None, None, :, :512].expand(1, H, T, 512),
        is_causal=True, scale=inp.softmax_scale)
    got = torch.from_numpy(out.reshape(T, H, 512)).permute(1, 0, 2)
    torch.testing.assert_close(got, ref[0], rtol=0, atol=1e-12)


def test_single_key_returns_v_exactly():
    """L = 0, T = 1: the only visible key is the token itself, so out is its V
    row exactly and lse is its one scaled score."""
    inp = make_inputs(batch=3, num_heads=4, prefix=[0, 0, 0], T=1, tree="chain",
                      pool_slots=128, nsplit=4, seed=23)
    out, lse = _oracle(inp)
    for b in range(3):
        krow = bf16_bits_to_f32(inp.kv_pool[inp.out_cache_loc[b]]).astype(np.float64)
        for h in range(4):
            n = b * 4 + h
            assert np.array_equal(out[n], krow[:512])
            qrow = bf16_bits_to_f32(inp.q[b, h]).astype(np.float64)
            assert abs(lse[n] - inp.softmax_scale * float(np.dot(qrow, krow))) < 1e-12


def test_zero_query_closed_form():
    """q = 0: all visible scores are 0, so out = mean of the visible V rows and
    lse = ln |visible| with |visible| = L_b + depth(t) + 1."""
    inp = make_inputs(batch=2, num_heads=2, prefix=[13, 4], T=8, tree="random", pool_slots=512,
                      nsplit=4, seed=24, q_mode="zero")
    out, lse = _oracle(inp)
    for b in range(2):
        for t in range(8):
            depth, v = 0, int(inp.tree_parent[b, t])
            while v != -1:
                depth, v = depth + 1, int(inp.tree_parent[b, v])
            nvis = int(inp.prefix_lens[b]) + depth + 1
            slots = visible_slots(inp, b, t)
            assert len(slots) == nvis
            mean = bf16_bits_to_f32(inp.kv_pool[slots])[:, :512].astype(np.float64).mean(axis=0)
            for h in range(2):
                n = (b * 8 + t) * 2 + h
                np.testing.assert_allclose(out[n], mean, rtol=0, atol=1e-12)
                assert abs(lse[n] - np.log(nvis)) < 1e-12


def test_placement_invariance_exact():
    """Scattered vs contiguous slots with the same logical content give
    identical results (the definition depends only on logical key order)."""
    a = make_inputs(batch=2, num_heads=2, prefix=[50, 70], T=8, tree="random", pool_slots=2000,
                    nsplit=4, seed=25, placement="scattered")
    c = make_inputs(batch=2, num_heads=2, prefix=[50, 70], T=8, tree="random", pool_slots=2000,
                    nsplit=4, seed=25, placement="contiguous")
    assert not np.array_equal(a.out_cache_loc, c.out_cache_loc)
    oa, la = _oracle(a)
    oc, lc = _oracle(c)
    assert np.array_equal(oa, oc) and np.array_equal(la, lc)


def test_request_independence_exact():
    """A batched call equals separate one-request calls, row for row."""
    inp = make_inputs(batch=3, num_heads=2, prefix=[9, 0, 30], T=4, tree="random",
                      pool_slots=1024, nsplit=2, seed=26)
    out, lse = _oracle(inp)
    per = inp.T * inp.num_heads
    for b in range(3):
        sub = make_inputs(batch=1, num_heads=2, prefix=[int(inp.prefix_lens[b])], T=4,
                          tree=inp.tree_parent[b:b + 1], pool_slots=1024, nsplit=2, seed=26)
        sub.q = inp.q[b * 4:(b + 1) * 4].copy()
        sub.kv_pool = inp.kv_pool
        sub.req_to_token = inp.req_to_token
        sub.req_pool_indices = inp.req_pool_indices[b:b + 1].copy()
        sub.out_cache_loc = inp.out_cache_loc[b * 4:(b + 1) * 4].copy()
        o, l = _oracle(sub)
        assert np.array_equal(o, out[b * per:(b + 1) * per])
        assert np.array_equal(l, lse[b * per:(b + 1) * per])


def test_head_permutation_exact():
    inp = make_inputs(batch=1, num_heads=4, prefix=[20], T=4, tree="random", pool_slots=256,
                      nsplit=2, seed=27)
    out, lse = _oracle(inp)
    perm = np.array([2, 0, 3, 1])
    inp2 = make_inputs(batch=1, num_heads=4, prefix=[20], T=4, tree="random", pool_slots=256,
                       nsplit=2, seed=27)
    inp2.q = inp.q[:, perm].copy()
    out2, lse2 = _oracle(inp2)
    o = out.reshape(4, 4, 512)
    o2 = out2.reshape(4, 4, 512)
    assert np.array_equal(o2, o[:, perm])
    assert np.array_equal(lse2.reshape(4, 4), lse.reshape(4, 4)[:, perm])


def test_scale_enters_the_scores():
    """Doubling q (exact in bf16) and halving the scale leaves the scores, and so
    the result, unchanged up to rounding; the unscaled case differs."""
    inp = make_inputs(batch=1, num_heads=2, prefix=[40], T=4, tree="random", pool_slots=256,
                      nsplit=2, seed=28)
    out, lse = _oracle(inp)
    q2 = inp.q.copy()
    nz = (q2 & 0x7F80) != 0  # normal numbers: add one to the exponent
    q2[nz] = q2[nz] + 0x0080
    inp2 = make_inputs(batch=1, num_heads=2, prefix=[40], T=4, tree="random", pool_slots=256,
                       nsplit=2, seed=28, softmax_scale=inp.softmax_scale / 2)
    inp2.q = q2
    out2, lse2 = _oracle(inp2)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    inp3 = make_inputs(batch=1, num_heads=2, prefix=[40], T=4, tree="random", pool_slots=256,
                       nsplit=2, seed=28, softmax_scale=1.0)
    _, lse3 = _oracle(inp3)
    assert np.abs(lse3 - lse).max() > 1e-3


def test_row_subset_matches_full():
    inp = make_config(1)
    out, lse = _oracle(inp)
    rows = [31, 0, 17, 5]
    o, l = _oracle(inp, rows=rows)
    assert np.array_equal(o, out[rows]) and np.array_equal(l, lse[rows])


def test_lse_is_natural_log_of_partition_sum():
    """Brute check of the LSE convention on one row: exp(lse) equals the sum of
    exp(scaled score) over the visible keys."""
    inp = make_inputs(batch=1, num_heads=1, prefix=[6], T=3, tree="chain", pool_slots=64,
                      nsplit=1, seed=29)
    _, lse = _oracle(inp)
    q = bf16_bits_to_f32(inp.q[2, 0]).astype(np.float64)
    s = [inp.softmax_scale * float(np.dot(q, bf16_bits_to_f32(inp.kv_pool[k]).astype(np.float64)))
         for k in visible_slots(inp, 0, 2)]
    assert abs(np.exp(lse[2]) - sum(np.exp(x) for x in s)) < 1e-9 * np.exp(lse[2])


def test_invalid_tree_is_rejected():
    inp = make_inputs(batch=1, num_heads=1, prefix=[4], T=3, tree=[-1, 2, 0], pool_slots=64,
                      nsplit=1, seed=30)
    with pytest.raises(ValueError):
        oracle.build_meta(inp)


def test_all_small_trees_brute_force():
    """Every parent array for T = 4 (3! = 6 trees): oracle == brute force."""
    T = 4
    for choice in itertools.product(*[range(i) for i in range(1, T)]):
        par = [-1] + list(choice)
        inp = make_inputs(batch=1, num_heads=1, prefix=[3], T=T, tree=par, pool_slots=32,
                          nsplit=1, seed=31)
        out, lse = _oracle(inp)
        for n in range(T):
            bo, bl = brute_row(inp, n)
            np.testing.assert_allclose(out[n], bo, rtol=0, atol=1e-12)
            assert abs(lse[n] - bl) <= 1e-12
