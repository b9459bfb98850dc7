"""GPU index/mask builder: bit-exact against the oracle's builder."""

import itertools

import numpy as np
import pytest
import torch

import mla_speculative_decoding_gb300 as mv
import oracle
from tests.gpu_util import config_cached, run_gpu, status
from workloads import make_config, make_inputs

pytestmark = pytest.mark.gpu


def _gpu_meta(inp, capacity=None):
    d = mv.to_device(inp, capacity=capacity)
    d.build()
    torch.cuda.synchronize()
    return (d.kv_indptr.cpu().numpy(), d.kv_indices.cpu().numpy(),
            d.anc_mask.cpu().numpy().view(np.uint64).reshape(inp.batch, inp.T), status(d))


def _check_exact(inp):
    ip, ix, anc = oracle.build_meta(inp)
    gip, gix, ganc, st = _gpu_meta(inp)
    assert st == 0
    assert np.array_equal(gip, ip)
    assert np.array_equal(gix[:len(ix)], ix)
    assert np.array_equal(ganc, anc)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_builder_configs_bit_exact(idx):
    _check_exact(make_config(idx))


@pytest.mark.parametrize("B,L", [(1, [0]), (2, [7, 0]), (8, [0, 1, 31, 32, 33, 1000, 5, 0])])
def test_builder_ragged_batches(B, L):
    _check_exact(make_inputs(batch=B, num_heads=1, prefix=L, T=9, tree="random",
                             pool_slots=4096, nsplit=4, seed=B))


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6])
def test_builder_every_tree_exhaustive(T):
    """All (T-1)! parent arrays at once, one request per tree."""
    trees = [[-1] + list(c) for c in itertools.product(*[range(i) for i in range(1, T)])]
    B = len(trees)
    inp = make_inputs(batch=B, num_heads=1, prefix=[3] * B, T=T, tree=np.array(trees),
                      pool_slots=8192, nsplit=2, seed=T)
    _check_exact(inp)


def test_builder_deterministic():
    inp = config_cached(5)
    a = _gpu_meta(inp)
    b = _gpu_meta(inp)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_builder_max_tree():
    inp = make_inputs(batch=3, num_heads=1, prefix=[10, 0, 70], T=64, tree="chain",
                      pool_slots=4096, nsplit=4, seed=6)
    _check_exact(inp)


def test_builder_capacity_truncates_and_flags():
    inp = make_inputs(batch=3, num_heads=1, prefix=[10, 20, 30], T=4, tree="random",
                      pool_slots=4096, nsplit=4, seed=7)
    ip, ix, _ = oracle.build_meta(inp)
    cap = 40  # fewer than the 72 keys
    gip, gix, _, st = _gpu_meta(inp, capacity=cap)
    assert st & mv.MLA_STATUS_CAPACITY
    assert gip.tolist() == [0, 14, 38, 40]
    assert np.array_equal(gix[:cap], ix[:cap])


def test_builder_bad_parent_is_root_and_flagged():
    inp = make_inputs(batch=1, num_heads=1, prefix=[5], T=4, tree=[-1, 0, 7, 1],
                      pool_slots=512, nsplit=2, seed=8)
    gip, gix, ganc, st = _gpu_meta(inp)
    assert st & mv.MLA_STATUS_BAD_PARENT
    assert [int(x) for x in ganc[0]] == [0b0001, 0b0011, 0b0100, 0b1011]


def test_builder_bad_table_row_flagged():
    inp = make_inputs(batch=2, num_heads=1, prefix=[5, 6], T=2, tree="chain",
                      pool_slots=512, nsplit=2, seed=9)
    inp.req_pool_indices = np.array([1, 9], dtype=np.int32)  # row 9 does not exist
    gip, gix, _, st = _gpu_meta(inp)
    assert st & mv.MLA_STATUS_BAD_PREFIX
    assert gip.tolist() == [0, 7, 9]  # request 1 keeps only its tree keys
    assert gix[7:9].tolist() == inp.out_cache_loc[2:4].tolist()
