"""The paged verify entry point (mla_verify_attention_paged): the partial
kernels read each key's pool slot from the page table and the draft slots
instead of a prebuilt combined list. On valid inputs it must give, bit for
bit, what the builder followed by the list-form attention gives, and so
match the oracle; bad table rows and prefixes are flagged and contained."""

import pytest
import torch

import mla_speculative_decoding_gb300 as mv
from tests.gpu_util import compare, config_cached, host_out, oracle_ref, sample_rows, status
from workloads import make_inputs
from workloads.gen import make_sparse_decode

pytestmark = pytest.mark.gpu


def _both(inp):
    """(list form: build + attention from tree_parent, paged form) outputs."""
    d = mv.to_device(inp)
    d.build()
    d.attention(use_anc=False)
    torch.cuda.synchronize()
    ref = (d.out.clone(), d.lse.clone(), status(d))
    d.workspace[:256].zero_()
    d.out.zero_()
    d.lse.zero_()
    d.step_paged()
    torch.cuda.synchronize()
    return ref, (d.out.clone(), d.lse.clone(), status(d)), d


def _bit_equal(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_paged_bit_identical_to_built_list(idx):
    (o1, l1, s1), (o2, l2, s2), _ = _both(config_cached(idx))
    assert s1 == 0 and s2 == 0
    assert _bit_equal(o1, o2) and _bit_equal(l1, l2)


def test_paged_sparse_decode_bit_identical():
    (o1, l1, s1), (o2, l2, s2), _ = _both(make_sparse_decode())
    assert s1 == 0 and s2 == 0
    assert _bit_equal(o1, o2) and _bit_equal(l1, l2)


CASES = [
    (1, 8, [1000], 16, "random", 7),
    (3, 8, [0, 129, 5], 16, "star", 64),
    (4, 32, [64, 0, 1, 4000], 4, "random", 16),
    (3, 8, [0, 129, 5], 33, "star", 64),
    (1, 64, [0], 64, "chain", 4),
    (6, 32, [1500, 0, 17, 4000, 260, 2500], 16, "random", 8),
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_paged_edge_cases(case):
    B, H, L, T, tree, ns = case
    inp = make_inputs(batch=B, num_heads=H, prefix=L, T=T, tree=tree,
                      pool_slots=max(16384, 2 * (sum(L) + B * T)), nsplit=ns, seed=sum(L) + T)
    (o1, l1, s1), (o2, l2, s2), d = _both(inp)
    assert s1 == 0 and s2 == 0
    assert _bit_equal(o1, o2) and _bit_equal(l1, l2)
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, f"paged case {case}")


def test_paged_long_workload_oracle_sampled():
    inp = config_cached(4)
    d = mv.to_device(inp)
    d.step_paged()
    torch.cuda.synchronize()
    assert status(d) == 0
    out, lse = host_out(d)
    rows = sample_rows(inp, per_request=12, seed=11)
    ref_out, ref_lse = oracle_ref(inp, rows=rows)
    compare(out[rows], lse[rows], ref_out, ref_lse, "paged long")


def test_paged_bad_rows_flagged_and_contained():
    """A table row outside the table and a prefix longer than the row are
    clamped as the builder clamps them (the request keeps only its draft
    keys, resp. the whole row) and flagged MLA_STATUS_BAD_PREFIX; the other
    requests' outputs are bit-identical to the builder path's and every
    output stays finite."""
    inp = make_inputs(batch=3, num_heads=8, prefix=[300, 200, 100], T=8, tree="random",
                      pool_slots=16384, nsplit=8, seed=7)
    d = mv.to_device(inp)
    d.build()
    d.attention(use_anc=False)
    torch.cuda.synchronize()
    o_ok = d.out[:8].clone()  # request 0's rows (T = 8, H = 8)
    l_ok = d.lse[:8].clone()
    stride = d.req_to_token.shape[1]
    d.req_pool_indices[1] = d.req_to_token.shape[0] + 5  # no such row
    d.prefix_lens[2] = stride + 50                       # longer than a row
    d.workspace[:256].zero_()
    d.step_paged()
    torch.cuda.synchronize()
    assert status(d) & mv.MLA_STATUS_BAD_PREFIX
    assert _bit_equal(o_ok, d.out[:8]) and _bit_equal(l_ok, d.lse[:8])
    assert torch.isfinite(d.out.float()).all() and not torch.isnan(d.lse).any()


def test_paged_rejects_bad_arguments():
    inp = config_cached(1)
    d = mv.to_device(inp)
    with pytest.raises(RuntimeError):
        mv.mla_verify_attention_paged(d.q, d.kv_pool, d.req_to_token, d.req_pool_indices,
                                      d.prefix_lens, d.out_cache_loc, d.tree_parent, d.T, 0,
                                      d.workspace, d.out, d.lse, d.softmax_scale)


def test_paged_step_in_a_cuda_graph():
    """The paged call is capture-safe: a captured step replays to the eager
    result bit for bit (the benchmark times it this way too)."""
    inp = config_cached(2)
    d = mv.to_device(inp)
    d.step_paged()
    torch.cuda.synchronize()
    o_ref, l_ref = d.out.clone(), d.lse.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d.step_paged()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        d.step_paged()
    d.out.zero_()
    d.lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert status(d) == 0
    assert _bit_equal(o_ref, d.out) and _bit_equal(l_ref, d.lse)
