"""GPU parity of the decode steps beside the verify attention (greedy tree
acceptance, KV relocation, fp8 paged indexer) and of the sparse-MLA decode
workload, against the CPU oracle, through the C ABI. Integer work is
bit-exact; the indexer's fp32 logits are within 1e-4 relative of the fp64
oracle (fp32 accumulation of 128 exact fp8 products per head)."""

import numpy as np
import pytest
import torch

import mla_speculative_decoding_gb300 as mv
import oracle
from tests.gpu_util import compare, host_out, oracle_ref, run_gpu, status
from workloads import (make_accept_inputs, make_indexer_inputs, make_inputs,
                       make_relocate_inputs, make_sparse_decode)

pytestmark = pytest.mark.gpu


def _dev(a, dtype=torch.int32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------- tree acceptance
def _accept_gpu(x, stream=None):
    B, T = x.tree_parent.shape
    outs = [torch.full((B,), -7, dtype=torch.int32, device="cuda")] + \
        [torch.full((B, T), -7, dtype=torch.int32, device="cuda") for _ in range(3)]
    st = _status()
    mv.mla_tree_accept(_dev(x.tree_parent), _dev(x.draft_tokens), _dev(x.target_argmax),
                       _dev(x.out_cache_loc), *outs, st, stream=stream)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs], int(st.item())


@pytest.mark.parametrize("T", [1, 2, 16, 31, 32, 33, 64])
@pytest.mark.parametrize("tree", ["random", "chain", "star"])
@pytest.mark.parametrize("match", [0.0, 0.6, 1.0])
def test_tree_accept_bit_exact(T, tree, match):
    x = make_accept_inputs(batch=9, T=T, tree=tree, vocab=5, match=match, seed=T + int(10 * match))
    got, st = _accept_gpu(x)
    ref = oracle.tree_accept(x.tree_parent, x.draft_tokens, x.target_argmax, x.out_cache_loc)
    assert st == 0
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_tree_accept_bad_parent_is_flagged_and_unreachable():
    x = make_accept_inputs(batch=2, T=8, tree="chain", vocab=3, match=1.0, seed=1)
    x.tree_parent = x.tree_parent.copy()
    x.tree_parent[1, 3] = 6          # not an earlier node: node 3 cannot be reached
    got, st = _accept_gpu(x)
    assert st & mv.MLA_STATUS_BAD_PARENT
    commit = got[0]
    assert commit[0] == 8 and commit[1] == 3   # request 1 stops before node 3
    r0 = oracle.tree_accept(x.tree_parent[:1], x.draft_tokens[:1], x.target_argmax[:1],
                            x.out_cache_loc[:1])
    for g, r in zip(got, r0):
        assert np.array_equal(g[:1], r)


# ---------------------------------------------------------------- KV relocation
def _reloc_state(x):
    pool = torch.from_numpy(x.kv_pool.view(np.int16)).cuda().view(torch.bfloat16)
    return dict(kv_pool=pool, req_to_token=_dev(x.req_to_token),
                req_pool_indices=_dev(x.req_pool_indices), prefix_lens=_dev(x.prefix_lens),
                dst_start=_dev(x.dst_start), progress=_dev(x.progress))


@pytest.mark.parametrize("budget", [1, 7, 64, 100_000])
def test_kv_relocate_matches_oracle_call_by_call(budget):
    x = make_relocate_inputs(batch=5, prefix=[300, 0, 1, 129, 64], pool_slots=4096, seed=budget,
                             in_place=5)
    d = _reloc_state(x)
    pool, r2t, prog = x.kv_pool, x.req_to_token, x.progress
    st = _status()
    for _ in range(400):
        if (prog >= x.prefix_lens).all():
            break
        mv.mla_kv_relocate(d["kv_pool"], d["req_to_token"], d["req_pool_indices"],
                           d["prefix_lens"], d["dst_start"], d["progress"], budget, st)
        pool, r2t, prog = oracle.kv_relocate(pool, r2t, x.req_pool_indices, x.prefix_lens,
                                             x.dst_start, prog, budget)
        torch.cuda.synchronize()
        assert np.array_equal(d["progress"].cpu().numpy(), prog)
        assert np.array_equal(d["req_to_token"].cpu().numpy(), r2t)
    got_pool = d["kv_pool"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_pool, pool)
    assert int(st.item()) == 0 and (prog == x.prefix_lens).all()


def test_kv_relocate_keeps_gpu_attention_bitwise_and_captures():
    """Relocating a verify workload's prefix rows into fresh contiguous slots
    (one captured CUDA-graph call replayed until done) leaves the GPU verify
    output bit-identical: the reduction order depends only on logical order."""
    L = [4000, 0, 1500]
    inp = make_inputs(batch=3, num_heads=16, prefix=L, T=16, tree="random", pool_slots=20000,
                      nsplit=16, seed=21, placement="contiguous")
    before = run_gpu(inp)
    o0 = before.out.cpu().view(torch.int16).numpy().copy()
    l0 = before.lse.cpu().numpy().copy()
    n = sum(L) + 3 * 16
    dst = (n + 100 + np.concatenate([[0], np.cumsum(L)[:-1]])).astype(np.int32)
    pool = before.kv_pool
    r2t = before.req_to_token
    rpi = _dev(inp.req_pool_indices)
    lens = _dev(inp.prefix_lens)
    dstd = _dev(dst)
    prog = torch.zeros(3, dtype=torch.int32, device="cuda")
    st = _status()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        mv.mla_kv_relocate(pool, r2t, rpi, lens, dstd, prog, 512, st, stream=s)  # warm-up call
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        mv.mla_kv_relocate(pool, r2t, rpi, lens, dstd, prog, 512, st)
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize()
    assert prog.cpu().tolist() == L and int(st.item()) == 0
    table = r2t.cpu().numpy()
    for b in range(3):
        assert table[inp.req_pool_indices[b], :L[b]].tolist() == list(range(dst[b], dst[b] + L[b]))
    before.step()
    torch.cuda.synchronize()
    assert np.array_equal(before.out.cpu().view(torch.int16).numpy(), o0)
    assert np.array_equal(before.lse.cpu().numpy(), l0)


def test_kv_relocate_bad_slot_is_flagged():
    x = make_relocate_inputs(batch=2, prefix=[10, 10], pool_slots=256, seed=3)
    x.dst_start = x.dst_start.copy()
    x.dst_start[1] = 250             # rows 6.. of request 1 fall outside the pool
    d = _reloc_state(x)
    st = _status()
    mv.mla_kv_relocate(d["kv_pool"], d["req_to_token"], d["req_pool_indices"], d["prefix_lens"],
                       d["dst_start"], d["progress"], 100, st)
    torch.cuda.synchronize()
    assert int(st.item()) & mv.MLA_STATUS_BAD_SLOT
    row = d["req_to_token"].cpu().numpy()[x.req_pool_indices[1]]
    assert row[:6].tolist() == list(range(250, 256))
    assert (row[6:10] == x.req_to_token[x.req_pool_indices[1], 6:10]).all()  # untouched


# ---------------------------------------------------------------- sparse-MLA decode
def test_sparse_decode_workload():
    inp = make_sparse_decode()
    d = run_gpu(inp)
    assert status(d) == 0
    out, lse = host_out(d)
    rows = np.arange(0, inp.num_rows, 3)
    ref_out, ref_lse = oracle_ref(inp, rows=rows)
    compare(out[rows], lse[rows], ref_out, ref_lse, "sparse decode")


@pytest.mark.parametrize("flags", [0, mv.MLA_PARTIAL_QUAD])
def test_sparse_decode_small_batch_full(flags):
    inp = make_sparse_decode(batch=2, pool_slots=20000, seed=9)
    d = run_gpu(inp, flags=flags)
    out, lse = host_out(d)
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, f"sparse decode flags {flags}")


# ---------------------------------------------------------------- fp8 indexer
def _indexer_gpu(ix, stream=None):
    B, P = ix.block_table.shape
    out = torch.full((B, P * 64), 123.0, dtype=torch.float32, device="cuda")
    st = _status()
    mv.mla_fp8_indexer_logits(_dev(ix.q, torch.uint8), _dev(ix.weights, torch.float32),
                              _dev(ix.kv_blocks, torch.uint8), _dev(ix.block_table),
                              _dev(ix.seq_lens), out, st, stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), int(st.item())


def _indexer_close(got, ref):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin) and np.isneginf(got[~fin]).all()
    if fin.any():
        scale = np.abs(ref[fin]).max()
        err = np.abs(got[fin] - ref[fin])
        assert (err <= 1e-4 * np.abs(ref[fin]) + 1e-5 * scale).all(), err.max()


@pytest.mark.parametrize("H", [1, 16, 64, 128])
@pytest.mark.parametrize("lens", [[1, 63, 64, 65], [0, 700, 129, 3000]])
def test_fp8_indexer_matches_oracle(H, lens):
    P = max((max(lens) + 63) // 64, 1) + 2       # pages past every request
    ix = make_indexer_inputs(batch=len(lens), num_heads=H, seq_lens=lens, max_pages=P,
                             seed=H + sum(lens))
    got, st = _indexer_gpu(ix)
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table, ix.seq_lens)
    assert st == 0
    _indexer_close(got, ref)


@pytest.mark.parametrize("H", [1, 20, 100])
def test_fp8_indexer_odd_pages_and_lengths_past_the_table(H):
    """Seven pages: the last 128-position tile holds a single page; the third
    request is longer than the table, so only its first 448 positions exist."""
    ix = make_indexer_inputs(batch=3, num_heads=H, seq_lens=[64 * 7, 64 * 5 + 3, 1000],
                             max_pages=16, seed=30 + H)
    ix.block_table = np.ascontiguousarray(ix.block_table[:, :7])
    got, st = _indexer_gpu(ix)
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table, ix.seq_lens)
    assert st == 0 and got.shape == (3, 448)
    _indexer_close(got, ref)


def test_fp8_indexer_many_short_requests():
    """300 requests of mixed short lengths (zeros included): each CTA's share
    spans many requests, so query tiles are reloaded and both query buffers
    recycled many times."""
    rng = np.random.default_rng(22)
    lens = rng.choice([0, 1, 63, 64, 65, 127, 128, 129, 500, 2000], size=300).astype(np.int32)
    ix = make_indexer_inputs(batch=300, num_heads=64, seq_lens=lens, max_pages=33, seed=22)
    got, st = _indexer_gpu(ix)
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table, ix.seq_lens)
    assert st == 0
    _indexer_close(got, ref)


def test_fp8_indexer_long_requests_span_several_windows():
    """4 requests x 160k positions (5000 tiles): every CTA walks more than 32
    tiles, crossing producer windows and ring laps; one head keeps the
    oracle fast."""
    ix = make_indexer_inputs(batch=4, num_heads=1, seq_lens=[160_000, 159_999, 100_001, 160_000],
                             max_pages=2500, seed=23)
    got, st = _indexer_gpu(ix)
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table, ix.seq_lens)
    assert st == 0
    _indexer_close(got, ref)


def test_fp8_indexer_timed_workload_sampled_pages():
    """The timed shape (16 requests x 32768 positions, 64 heads, 4097-page
    table): every position past the lengths is -inf, and two random full
    pages per request match the oracle run on just those pages (the logits
    of a page depend only on its block, the request's queries and weights)."""
    ix = make_indexer_inputs(batch=16, num_heads=64, seq_lens="fixed:32768", max_pages=4097,
                             seed=13)
    got, st = _indexer_gpu(ix)
    assert st == 0
    assert np.isneginf(got[:, 32768:]).all() and np.isfinite(got[:, :32768]).all()
    rng = np.random.default_rng(24)
    pages = np.stack([rng.choice(512, size=2, replace=False) for _ in range(16)]).astype(np.int64)
    bt = np.take_along_axis(ix.block_table, pages, axis=1).astype(np.int32)
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, bt,
                                    np.full(16, 128, np.int32))
    sub = np.stack([np.concatenate([got[b, 64 * p:64 * p + 64] for p in pages[b]])
                    for b in range(16)])
    _indexer_close(sub, ref)


def test_fp8_indexer_bad_block_is_flagged_and_graph_capturable():
    ix = make_indexer_inputs(batch=2, num_heads=64, seq_lens=[200, 100], max_pages=4, seed=4)
    ix.block_table = ix.block_table.copy()
    ix.block_table[1, 1] = 99_999
    got, st = _indexer_gpu(ix)
    assert st & mv.MLA_STATUS_BAD_SLOT
    assert np.isneginf(got[1, 64:128]).all()
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks,
                                    np.where(ix.block_table < ix.kv_blocks.shape[0], ix.block_table, -1),
                                    np.array([200, 64], np.int32))
    _indexer_close(got[0], ref[0])
    _indexer_close(got[1, :64], ref[1, :64])
    # capture in a CUDA graph: the fixed grid replays and follows new lengths
    ix = make_indexer_inputs(batch=3, num_heads=64, seq_lens=[300, 200, 128], max_pages=6, seed=8)
    q, w, kv = _dev(ix.q, torch.uint8), _dev(ix.weights, torch.float32), _dev(ix.kv_blocks, torch.uint8)
    bt, sl = _dev(ix.block_table), _dev(np.array([300, 5, 128], np.int32))
    out = torch.zeros(3, 6 * 64, dtype=torch.float32, device="cuda")
    st = _status()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mv.mla_fp8_indexer_logits(q, w, kv, bt, sl, out, st, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mv.mla_fp8_indexer_logits(q, w, kv, bt, sl, out, st)
    sl.copy_(torch.tensor([100, 200, 0], dtype=torch.int32))
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.fp8_indexer_logits(ix.q, ix.weights, ix.kv_blocks, ix.block_table,
                                    np.array([100, 200, 0], np.int32))
    _indexer_close(out.cpu().numpy().astype(np.float64), ref)
