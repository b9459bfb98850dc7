"""Checks of the seeded input generator (shapes, determinism, placement)."""

import numpy as np

from workloads import CONFIGS, bf16_bits_to_f32, f32_to_bf16_bits, make_config, make_inputs


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-39], dtype=np.float32)
    b = f32_to_bf16_bits(x)
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1.0); 1+3*2^-8 ties up to 1+2^-6.
    assert bf16_bits_to_f32(b).tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5,
                                            float(bf16_bits_to_f32(b[4:5])[0])]
    assert b[0] == 0x3F80 and b[3] == 0xC020


def test_deterministic_and_seed_sensitive():
    a = make_inputs(batch=2, num_heads=2, prefix="uniform:5:9", T=4, pool_slots=128, seed=7)
    b = make_inputs(batch=2, num_heads=2, prefix="uniform:5:9", T=4, pool_slots=128, seed=7)
    c = make_inputs(batch=2, num_heads=2, prefix="uniform:5:9", T=4, pool_slots=128, seed=8)
    for f in ("prefix_lens", "tree_parent", "req_to_token", "out_cache_loc", "q", "kv_pool"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert not np.array_equal(a.q, c.q)


def test_tiny_config_shapes_and_poison():
    inp = make_config(1)
    assert inp.q.shape == (4, 8, 576) and inp.kv_pool.shape == (4096, 576)
    assert inp.tree_parent.tolist() == [[-1, 0, 1, 2]]
    used = set(inp.req_to_token[inp.req_pool_indices[0], :256].tolist()) | set(
        inp.out_cache_loc.tolist())
    assert len(used) == 260
    unused = np.setdiff1d(np.arange(4096), np.array(sorted(used)))
    assert np.all(inp.kv_pool[unused] == 0x7FC0)
    assert np.all(np.isfinite(bf16_bits_to_f32(inp.kv_pool[sorted(used)])))


def test_random_tree_parents_are_earlier_nodes():
    inp = make_inputs(batch=4, num_heads=1, prefix=[1, 2, 3, 4], T=16, pool_slots=256, seed=9)
    for b in range(4):
        assert inp.tree_parent[b, 0] == -1
        assert all(0 <= inp.tree_parent[b, i] < i for i in range(1, 16))


def test_contiguous_placement_keeps_logical_content():
    s = make_inputs(batch=2, num_heads=1, prefix=[10, 3], T=2, pool_slots=64, seed=5)
    c = make_inputs(batch=2, num_heads=1, prefix=[10, 3], T=2, pool_slots=64, seed=5,
                    placement="contiguous")
    assert np.array_equal(s.q, c.q)
    assert c.out_cache_loc.tolist() == [10, 11, 15, 16]
    r = c.req_pool_indices
    assert c.req_to_token[r[0], :10].tolist() == list(range(10))
    assert c.req_to_token[r[1], :3].tolist() == [12, 13, 14]
    # Same values at the same logical positions.
    assert np.array_equal(s.kv_pool[s.out_cache_loc], c.kv_pool[c.out_cache_loc])


def test_config_table():
    assert CONFIGS[1]["seed"] == 0 and CONFIGS[1]["nsplit"] == 4
    assert CONFIGS[4]["pool_slots"] == 195_011 and CONFIGS[4]["T"] == 64
    assert CONFIGS[5]["batch"] == 8 and CONFIGS[5]["num_heads"] == 64
