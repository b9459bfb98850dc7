"""The allocation-free verify entry point (mla_verify_attention_noalloc).

It serves callers that cannot allocate device memory where they run the
verify step (for example inside a runtime that owns all device memory), so
it keeps its partial results in the library's fixed device scratch area
instead of a caller workspace. It launches the same kernels as the
workspace entry point, so this file checks, through the C ABI, that its
results are bit-identical to that entry point's on two calls in a row (the
second call reuses the scratch left by the first), at a shape just under
the scratch size, that it reports its own status bits only, and that
shapes just past the scratch size are refused before anything runs. It is
collected last on purpose.
"""

import pytest
import torch

import mla_speculative_decoding_gb300 as mv
from workloads import make_inputs

pytestmark = pytest.mark.gpu


def _case(seed, prefix, T, H, nsplit):
    inp = make_inputs(batch=len(prefix), num_heads=H, prefix=prefix, T=T, tree="random",
                      pool_slots=32768, nsplit=nsplit, seed=seed)
    d = mv.to_device(inp)
    d.build()
    d.attention(use_anc=False)  # the existing entry point, with a caller workspace
    torch.cuda.synchronize()
    return inp, d


def _noalloc(d, status=None):
    out = torch.full_like(d.out, float("nan"))
    lse = torch.full_like(d.lse, float("nan"))
    mv.mla_verify_attention_noalloc(d.q, d.kv_pool, d.kv_indices, d.kv_indptr, d.prefix_lens,
                                    d.tree_parent, d.T, d.nsplit, out, lse, d.softmax_scale,
                                    status=status)
    torch.cuda.synchronize()
    return out, lse


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                       b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


def _partials(inp):
    return inp.batch * inp.T * inp.num_heads * inp.nsplit


def test_noalloc_bit_identical_to_workspace_entry_point_twice():
    limit = mv.mla_verify_noalloc_scratch_bytes()
    cases = [_case(31, [5000, 777], 16, 8, 32), _case(32, [12000], 8, 16, 64),
             # 150 rows x 109 splits = 16,350 partials: just under the 32 MiB area
             _case(35, [3000], 10, 15, 109)]
    assert _partials(cases[-1][0]) == 16350
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for inp, d in cases:
        assert mv.mla_verify_workspace_bytes(inp.batch, inp.T, inp.num_heads, inp.nsplit) <= limit
        for _ in range(2):  # two calls in a row: the scratch keeps the last call's contents
            out, lse = _noalloc(d, status)
            assert _same_bits(out, d.out) and _same_bits(lse, d.lse)
            assert int(status.item()) == 0


def test_noalloc_status_reports_this_call_only():
    inp, d = _case(33, [900], 4, 8, 8)
    d.kv_indices[10] = 10 ** 8  # an out-of-range slot: flagged and masked
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _noalloc(d, status)
    assert int(status.item()) & mv.MLA_STATUS_BAD_SLOT
    inp2, d2 = _case(34, [900], 4, 8, 8)
    _noalloc(d2, status)
    assert int(status.item()) == 0  # the previous call's bits are not carried over


def _refused_shape(T, H, ns):
    q = torch.zeros(T, H, 576, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(16, 576, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(T + 2, dtype=torch.int32, device="cuda")
    par = torch.full((1, T), -1, dtype=torch.int32, device="cuda")
    out = torch.full((T, H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), 7.0, dtype=torch.float32, device="cuda")
    status = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    with pytest.raises(mv.MlaError) as e:
        mv.mla_verify_attention_noalloc(q, kv, i32, i32, i32, par, T, ns, out, lse, 0.07,
                                        status=status)
    torch.cuda.synchronize()
    # refused before anything was queued: outputs and status untouched
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all()) and int(status.item()) == 5
    return e.value.code


def test_noalloc_refuses_shapes_beyond_the_scratch():
    limit = mv.mla_verify_noalloc_scratch_bytes()
    assert limit == 32 << 20
    # 224 rows x 73 splits = 16,352 partials: one past what the area holds
    T, H, ns = 14, 16, 73
    assert mv.mla_verify_workspace_bytes(1, T, H, ns) > limit
    assert mv.mla_verify_workspace_bytes(1, 10, 15, 109) <= limit
    assert _refused_shape(T, H, ns) == -3
    # far beyond: 8192 rows x 128 splits
    assert _refused_shape(64, 128, 128) == -3
