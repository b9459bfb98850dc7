"""GPU verify attention vs the CPU fp64 oracle, element by element.

Every test calls the C ABI (through the thin binding) on seeded inputs and
compares with the oracle run on the same inputs. Both kernel paths are
covered: the default (the four-SM 2-SM-MMA kernel for requests of more
than 128 rows, the two-SM kernel otherwise), and each of the two forced.
"""

import numpy as np
import pytest
import torch

import mla_speculative_decoding_gb300 as mv
from tests.gpu_util import config_cached, compare, host_out, oracle_ref, run_gpu, sample_rows, status
from workloads import make_config, make_inputs

pytestmark = pytest.mark.gpu
PATHS = [0, mv.MLA_PARTIAL_PAIR, mv.MLA_PARTIAL_QUAD]


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("idx", [1, 2, 3])
def test_configs_full(idx, flags):
    inp = config_cached(idx)
    d = run_gpu(inp, flags=flags)
    assert status(d) == 0
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, f"config {idx} flags {flags}")


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("idx", [4, 5])
def test_configs_sampled_rows(idx, flags):
    """Full-size long/batched workloads in the benchmark's launch configuration;
    the oracle computes a sample of rows one by one."""
    inp = config_cached(idx)
    d = run_gpu(inp, flags=flags)
    assert status(d) == 0
    out, lse = host_out(d)
    rows = sample_rows(inp, per_request=12 if inp.batch == 1 else 6, seed=idx)
    ref_out, ref_lse = oracle_ref(inp, rows=rows)
    compare(out[rows], lse[rows], ref_out, ref_lse, f"config {idx} flags {flags}")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


@pytest.mark.parametrize("idx", [4, 5])
def test_configs_every_row_in_the_benchmark_call(idx):
    """The long and batched workloads at full size through the call the
    benchmark times (mla_verify_attention_paged): every output row and every
    lse against the oracle."""
    inp = config_cached(idx)
    d = mv.to_device(inp)
    d.step_paged()
    torch.cuda.synchronize()
    assert status(d) == 0
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, f"config {idx}, every row, paged call")


def test_config3_contiguous_placement():
    inp = config_cached(3, placement="contiguous")
    d = run_gpu(inp)
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, "config 3 contiguous")


CASES = [
    # (batch, heads, prefix, T, tree, nsplit)
    (1, 8, [1000], 16, "random", 7),        # ragged tail, odd split count
    (2, 16, [333, 2049], 8, "random", 5),   # ragged batch, 128 rows per request
    (1, 128, [700], 1, "chain", 3),         # maximum heads, single token
    (1, 2, [0], 64, "chain", 4),            # no prefix, maximum tree (causal)
    (3, 8, [0, 129, 5], 16, "star", 64),    # more splits than keys in some requests
    (1, 8, [300], 16, "random", 128),       # maximum split count
    (4, 32, [64, 0, 1, 4000], 4, "random", 16),
    # more than 128 rows per request: 256-row blocks, full and ragged
    (1, 16, [1000], 16, "random", 7),       # exactly one 256-row block
    (2, 8, [333, 2049], 24, "random", 5),   # 192 rows: second half of the block partly empty
    (1, 24, [700], 16, "random", 3),        # 384 rows: second block half empty
    (1, 128, [5000], 2, "chain", 9),        # 256 rows from 128 heads
    (3, 8, [0, 129, 5], 33, "star", 64),    # 264 rows: 8 rows in the last block; empty splits
    (1, 3, [2500], 43, "random", 11),       # 129 rows: one row past the two-SM kernel's range
    (1, 64, [0], 64, "chain", 4),           # 4096 rows, no prefix, maximum tree
    # more four-SM work items than resident clusters: each persistent cluster
    # walks several items of different requests, row blocks and lengths
    (6, 32, [1500, 0, 17, 4000, 260, 2500], 16, "random", 8),
    (2, 16, [20000, 100], 32, "random", 48),
    # more two-SM (request, row block) pairs than one wave of 76 clusters
    # holds: the wave-shaped split over several waves of partitions
    (96, 8, [(37 * k) % 1500 for k in range(96)], 4, "random", 8),
    (80, 4, [1200 + 13 * k for k in range(80)], 8, "random", 2),
]


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_edge_cases(case, flags):
    B, H, L, T, tree, ns = case
    inp = make_inputs(batch=B, num_heads=H, prefix=L, T=T, tree=tree,
                      pool_slots=max(16384, 2 * (sum(L) + B * T)), nsplit=ns, seed=sum(L) + T)
    d = run_gpu(inp, flags=flags)
    assert status(d) == 0
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, f"case {case} flags {flags}")


@pytest.mark.parametrize("flags", PATHS)
def test_single_key_returns_v_bit_exact(flags):
    """L = 0, T = 1: every head's output is the token's own V row, bit for bit."""
    inp = make_inputs(batch=4, num_heads=8, prefix=[0] * 4, T=1, tree="chain", pool_slots=256,
                      nsplit=4, seed=3)
    d = run_gpu(inp, flags=flags)
    got = d.out.cpu().view(torch.int16).numpy().view(np.uint16)
    for b in range(4):
        v = inp.kv_pool[inp.out_cache_loc[b], :512]
        for h in range(8):
            assert np.array_equal(got[b, h], v)
    _, ref_lse = oracle_ref(inp)
    _, lse = host_out(d)
    assert np.abs(lse - ref_lse).max() <= 1e-3


def test_zero_query_closed_form_on_gpu():
    inp = make_inputs(batch=2, num_heads=4, prefix=[500, 37], T=8, tree="random",
                      pool_slots=4096, nsplit=8, seed=4, q_mode="zero")
    d = run_gpu(inp)
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, "q = 0")


@pytest.mark.parametrize("heads", [4, 32])
@pytest.mark.parametrize("flags", PATHS)
def test_growing_scores_force_rescaling(flags, heads):
    """Scores that grow along the key order (about 48 nats over the prefix)
    make the running maximum overtake the lazy-rescale threshold (2^8, i.e.
    5.5 nats) many times. Magnitudes stay where fp32 scores can meet the 1e-3
    lse bound."""
    from workloads import bf16_bits_to_f32, f32_to_bf16_bits
    inp = make_inputs(batch=1, num_heads=heads, prefix=[3000], T=8, tree="random", pool_slots=4096,
                      nsplit=3, seed=41, placement="contiguous")
    q = np.abs(bf16_bits_to_f32(inp.q))
    inp.q = f32_to_bf16_bits(q)
    n = 3000 + 8
    kv = bf16_bits_to_f32(inp.kv_pool[:n]) + (0.0005 * np.arange(n, dtype=np.float32))[:, None]
    inp.kv_pool = inp.kv_pool.copy()
    inp.kv_pool[:n] = f32_to_bf16_bits(kv)
    d = run_gpu(inp, flags=flags)
    assert status(d) == 0
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, "growing scores")
