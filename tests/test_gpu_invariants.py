"""Invariants of the GPU verify path that must hold bit for bit (or within fp32
noise), CUDA-graph capture, and device status handling."""

import numpy as np
import pytest
import torch

import mla_speculative_decoding_gb300 as mv
from tests.gpu_util import compare, host_out, oracle_ref, run_gpu, status
from workloads import make_inputs

pytestmark = pytest.mark.gpu
PATHS = [0, mv.MLA_PARTIAL_PAIR, mv.MLA_PARTIAL_QUAD]


def _bits(d):
    return (d.out.cpu().view(torch.int16).numpy().copy(), d.lse.cpu().numpy().copy())


@pytest.mark.parametrize("T", [16, 40])
@pytest.mark.parametrize("flags", PATHS)
def test_placement_invariance_bitwise(flags, T):
    """Scattered vs contiguous slots (same logical content): identical bits,
    because the reduction order depends only on logical key order."""
    kw = dict(batch=2, num_heads=8, prefix=[9000, 3100], T=T, tree="random", pool_slots=60000,
              nsplit=64, seed=11)
    a = run_gpu(make_inputs(placement="scattered", **kw), flags=flags)
    c = run_gpu(make_inputs(placement="contiguous", **kw), flags=flags)
    oa, la = _bits(a)
    oc, lc = _bits(c)
    assert np.array_equal(oa, oc) and np.array_equal(la, lc)


@pytest.mark.parametrize("T", [8, 24])
@pytest.mark.parametrize("flags", PATHS)
def test_batch_equals_separate_calls_bitwise(flags, T):
    # A request's partitions may depend on the launch (the two-SM kernel's
    # one-wave split uses min(nsplit, resident clusters / pairs) of them):
    # nsplit 8 gives every request 8 in the batch and alone, and then the
    # results agree bit for bit.
    kw = dict(num_heads=8, T=T, tree="random", pool_slots=20000, nsplit=8, seed=12)
    inp = make_inputs(batch=3, prefix=[2000, 0, 777], **kw)
    d = run_gpu(inp, flags=flags)
    ob, lb = _bits(d)
    per = inp.T
    for b in range(3):
        sub = make_inputs(batch=1, prefix=[int(inp.prefix_lens[b])], **kw)
        sub.q = inp.q[b * per:(b + 1) * per].copy()
        sub.kv_pool = inp.kv_pool
        sub.tree_parent = inp.tree_parent[b:b + 1].copy()
        sub.req_to_token = inp.req_to_token
        sub.req_pool_indices = inp.req_pool_indices[b:b + 1].copy()
        sub.out_cache_loc = inp.out_cache_loc[b * per:(b + 1) * per].copy()
        o, l = _bits(run_gpu(sub, flags=flags))
        assert np.array_equal(o, ob[b * per:(b + 1) * per])
        assert np.array_equal(l, lb[b * per:(b + 1) * per])


@pytest.mark.parametrize("T", [8, 24])
@pytest.mark.parametrize("flags", PATHS)
def test_head_permutation_bitwise(flags, T):
    inp = make_inputs(batch=1, num_heads=16, prefix=[1500], T=T, tree="random", pool_slots=8192,
                      nsplit=8, seed=13)
    o, l = _bits(run_gpu(inp, flags=flags))
    perm = np.random.default_rng(0).permutation(16)
    inp.q = inp.q[:, perm].copy()
    o2, l2 = _bits(run_gpu(inp, flags=flags))
    assert np.array_equal(o2, o[:, perm]) and np.array_equal(l2, l[:, perm])


@pytest.mark.parametrize("T", [16, 48])
@pytest.mark.parametrize("flags", PATHS)
def test_inline_vs_prebuilt_mask_bitwise(flags, T):
    inp = make_inputs(batch=2, num_heads=8, prefix=[3000, 10], T=T, tree="random",
                      pool_slots=8192, nsplit=32, seed=14)
    a = _bits(run_gpu(inp, flags=flags, use_anc=True))
    b = _bits(run_gpu(inp, flags=flags, use_anc=False))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("T", [16, 32])
def test_split_count_invariance(T):
    inp = make_inputs(batch=1, num_heads=8, prefix=[6000], T=T, tree="random", pool_slots=8192,
                      nsplit=1, seed=15)
    res = {}
    for ns in (1, 4, 64):
        d = run_gpu(inp, nsplit=ns)
        res[ns] = host_out(d)
    for ns in (4, 64):
        assert np.max(np.abs(res[ns][1] - res[1][1]) / np.abs(res[1][1])) <= 1e-5
        assert np.max(np.abs(res[ns][0] - res[1][0])) <= 2e-2 * np.abs(res[1][0]).max()


@pytest.mark.parametrize("T", [16, 32])
@pytest.mark.parametrize("flags", PATHS)
def test_paths_agree(flags, T):
    inp = make_inputs(batch=2, num_heads=8, prefix=[5000, 1234], T=T, tree="random",
                      pool_slots=16384, nsplit=16, seed=16)
    out, lse = host_out(run_gpu(inp, flags=flags))
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("T", [16, 32])
def test_deterministic_repeat(T):
    inp = make_inputs(batch=2, num_heads=8, prefix=[5000, 1234], T=T, tree="random",
                      pool_slots=16384, nsplit=64, seed=17)
    d = run_gpu(inp)
    a = _bits(d)
    for _ in range(3):
        d.step()
        torch.cuda.synchronize()
        b = _bits(d)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("T", [16, 32])
def test_cuda_graph_capture_and_replay(T):
    """The whole verify step (build + partial + combine) is captured in one CUDA
    graph; replays match eager bit for bit and follow new input contents."""
    inp = make_inputs(batch=2, num_heads=8, prefix=[4000, 900], T=T, tree="random",
                      pool_slots=16384, nsplit=64, seed=18)
    d = run_gpu(inp)  # eager (also runs the one-time set-up outside capture)
    eager = _bits(d)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        d.step()  # warm-up on the side stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        d.step()
    d.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    rep = _bits(d)
    assert np.array_equal(rep[0], eager[0]) and np.array_equal(rep[1], eager[1])
    # New query contents in the same static buffer: the replay follows them.
    q2 = np.ascontiguousarray(inp.q[:, ::-1, :])
    d.q.copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    out, lse = host_out(d)
    inp.q = q2
    ref_out, ref_lse = oracle_ref(inp)
    compare(out, lse, ref_out, ref_lse, "graph replay with new q")


def test_capture_before_set_up_is_refused():
    """In a fresh process, a first call made inside stream capture (before the
    one-time set-up) returns MLA_ERR_NOT_INITIALIZED instead of running set-up
    during capture."""
    import subprocess
    import sys
    code = r"""
import torch, mla_speculative_decoding_gb300 as mv
from workloads import make_inputs
inp = make_inputs(batch=1, num_heads=8, prefix=[64], T=4, tree="chain", pool_slots=1024, nsplit=4, seed=1)
d = mv.to_device(inp)
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
code = None
try:
    with torch.cuda.graph(g):
        try:
            d.attention(use_anc=False)
        except mv.MlaError as e:
            code = e.code
except Exception:
    pass
print("CODE", code)
"""
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                       cwd=__import__("os").path.dirname(__import__("os").path.dirname(
                           __import__("os").path.abspath(__file__))))
    assert "CODE -5" in r.stdout, r.stdout + r.stderr


def test_bad_slot_is_masked_and_flagged():
    """An out-of-range slot: that key is masked (as if removed) and the status
    word says so."""
    inp = make_inputs(batch=1, num_heads=8, prefix=[700], T=8, tree="random", pool_slots=4096,
                      nsplit=8, seed=19)
    d = mv.to_device(inp)
    d.build()
    torch.cuda.synchronize()
    d.kv_indices[699] = 10 ** 6  # the last prefix key
    d.attention()
    torch.cuda.synchronize()
    assert status(d) & mv.MLA_STATUS_BAD_SLOT
    out, lse = host_out(d)
    ref = make_inputs(batch=1, num_heads=8, prefix=[700], T=8, tree="random", pool_slots=4096,
                      nsplit=8, seed=19)
    ref.prefix_lens = np.array([699], dtype=np.int32)
    ref.req_to_token = ref.req_to_token.copy()
    ref_out, ref_lse = oracle_ref(ref)
    compare(out, lse, ref_out, ref_lse, "masked bad slot")
    mv.mla_verify_reset_status(d.status)
    torch.cuda.synchronize()
    assert status(d) == 0


def test_bad_parent_node_is_a_root_and_flagged():
    """Inline mask from tree_parent: a node with an invalid parent sees only the
    prefix and itself; same as the prebuilt mask."""
    inp = make_inputs(batch=1, num_heads=4, prefix=[300], T=3, tree=[-1, 0, 9], pool_slots=4096,
                      nsplit=4, seed=20)
    d = mv.to_device(inp)
    d.build()
    d.attention(use_anc=False)
    torch.cuda.synchronize()
    assert status(d) & mv.MLA_STATUS_BAD_PARENT
    out, lse = host_out(d)
    # Node 2 behaves like a single-token request on its own slot.
    one = make_inputs(batch=1, num_heads=4, prefix=[300], T=1, tree="chain", pool_slots=4096,
                      nsplit=4, seed=20)
    one.kv_pool = inp.kv_pool
    one.req_to_token = inp.req_to_token
    one.req_pool_indices = inp.req_pool_indices
    one.out_cache_loc = inp.out_cache_loc[2:3].copy()
    one.q = inp.q[2:3].copy()
    ref_out, ref_lse = oracle_ref(one)
    compare(out[8:12], lse[8:12], ref_out, ref_lse, "bad parent root")


def test_inconsistent_indptr_flagged():
    inp = make_inputs(batch=1, num_heads=2, prefix=[100], T=4, tree="chain", pool_slots=1024,
                      nsplit=4, seed=21)
    d = mv.to_device(inp)
    d.build()
    torch.cuda.synchronize()
    d.kv_indptr[1] = 102  # two tree keys missing
    d.attention()
    torch.cuda.synchronize()
    assert status(d) & mv.MLA_STATUS_BAD_INDPTR
    out, lse = host_out(d)
    assert np.all(np.isfinite(out[:4])) and np.all(np.isfinite(lse[:4]))


def test_workspace_too_small_is_refused():
    inp = make_inputs(batch=1, num_heads=8, prefix=[64], T=4, tree="chain", pool_slots=1024,
                      nsplit=4, seed=22)
    d = mv.to_device(inp)
    with pytest.raises(mv.MlaError) as e:
        mv.mla_verify_attention(d.q, d.kv_pool, d.kv_indices, d.kv_indptr, d.prefix_lens,
                                d.tree_parent, d.T, d.nsplit, d.workspace[:-256], d.out, d.lse,
                                d.softmax_scale)
    assert e.value.code == -3
