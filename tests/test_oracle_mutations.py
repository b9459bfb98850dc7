"""Planted mistakes in the oracle are caught by its pins.

Each case copies the oracle's C source, plants one plausible slip by text
substitution, compiles the copy on the CPU, and runs a battery of the pins
(brute force on tiny inputs, the single-key V case, the zero-query closed
form, the chain = causal library case). The untouched source must pass the
battery and every planted slip must fail it.
"""

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from tests.brute import brute_row, visible_slots
from workloads import bf16_bits_to_f32, make_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "mla_verify_oracle.c")).read()

MUTATIONS = {
    "no_self_visibility": ("for (int v = t; v != -1; v = par[v])",
                           "for (int v = par[t]; v != -1; v = par[v])"),
    "v_from_wrong_dims": ("out_row[d] += w * bf16_to_double(k[d]);",
                          "out_row[d] += w * bf16_to_double(k[d + 64]);"),
    "scale_dropped": ("s_buf[i] = scale * acc;", "s_buf[i] = acc;"),
    "lse_log2": ("*lse_out = m + log(Z);", "*lse_out = m + log2(Z);"),
    "last_prefix_key_dropped": ("for (int32_t j = 0; j < Lb; ++j) key_buf[nvis++] = j;",
                                "for (int32_t j = 0; j + 1 < Lb; ++j) key_buf[nvis++] = j;"),
    "tree_slots_reversed": ("dst[prefix_lens[b] + u] = out_cache_loc[(int64_t)b * T + u];",
                            "dst[prefix_lens[b] + u] = out_cache_loc[(int64_t)b * T + (T - 1 - u)];"),
    "not_normalised": ("for (int d = 0; d < D_V; ++d) out_row[d] /= Z;", ""),
    "rope_dims_dropped": ("for (int d = 0; d < D_QK; ++d) acc += qd[d] * bf16_to_double(k[d]);",
                          "for (int d = 0; d < D_V; ++d) acc += qd[d] * bf16_to_double(k[d]);"),
}

_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)


def _compile(src, tmp_path, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_build_meta.argtypes = [_i32p, ctypes.c_int64, _i32p, _i32p, _i32p, _i32p,
                                      ctypes.c_int, ctypes.c_int, _i32p, _i32p, _u64p]
    lib.oracle_verify_attention.argtypes = [_u16p, _u16p, ctypes.c_int64, _i32p, _i32p, _i32p,
                                            _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, _i64p, ctypes.c_int64, _f64p, _f64p,
                                            ctypes.c_int]
    return lib


def _run(lib, inp):
    B, T = inp.batch, inp.T
    p = lambda a, t: a.ctypes.data_as(t)  # noqa: E731
    L = np.ascontiguousarray(inp.prefix_lens, np.int32)
    n = int(L.sum() + B * T)
    indptr = np.zeros(B + 1, np.int32)
    idx = np.zeros(max(n, 1), np.int32)
    anc = np.zeros(B * T, np.uint64)
    par = np.ascontiguousarray(inp.tree_parent, np.int32)
    r2t = np.ascontiguousarray(inp.req_to_token, np.int32)
    rc = lib.oracle_build_meta(p(r2t, _i32p), r2t.shape[1], p(inp.req_pool_indices, _i32p),
                               p(L, _i32p), p(inp.out_cache_loc, _i32p), p(par, _i32p), B, T,
                               p(indptr, _i32p), p(idx, _i32p), p(anc, _u64p))
    assert rc == 0
    out = np.zeros((inp.num_rows, 512))
    lse = np.zeros(inp.num_rows)
    rc = lib.oracle_verify_attention(p(inp.q, _u16p), p(inp.kv_pool, _u16p), inp.kv_pool.shape[0],
                                     p(idx, _i32p), p(indptr, _i32p), p(L, _i32p), p(par, _i32p),
                                     B, T, inp.num_heads, inp.softmax_scale, None, inp.num_rows,
                                     p(out, _f64p), p(lse, _f64p), 1)
    assert rc == 0
    return out, lse


def _battery(lib):
    """Returns the names of the pins that fail for this oracle build."""
    failed = []
    # Brute force on a tiny random-tree batch.
    inp = make_inputs(batch=2, num_heads=2, prefix=[5, 3], T=4, tree="random", pool_slots=64,
                      nsplit=2, seed=41)
    out, lse = _run(lib, inp)
    ok = True
    for n in range(inp.num_rows):
        bo, bl = brute_row(inp, n)
        ok &= bool(np.allclose(out[n], bo, rtol=0, atol=1e-12) and abs(lse[n] - bl) <= 1e-12)
    if not ok:
        failed.append("brute_force")
    # Single key: out is V exactly.
    inp = make_inputs(batch=1, num_heads=2, prefix=[0], T=1, tree="chain", pool_slots=16,
                      nsplit=1, seed=42)
    out, _ = _run(lib, inp)
    v = bf16_bits_to_f32(inp.kv_pool[inp.out_cache_loc[0]])[:512].astype(np.float64)
    if not (np.array_equal(out[0], v) and np.array_equal(out[1], v)):
        failed.append("single_key")
    # Zero query: mean of visible V rows, lse = ln |visible|.
    inp = make_inputs(batch=1, num_heads=1, prefix=[6], T=4, tree="random", pool_slots=64,
                      nsplit=1, seed=43, q_mode="zero")
    out, lse = _run(lib, inp)
    for t in range(4):
        s = visible_slots(inp, 0, t)
        mean = bf16_bits_to_f32(inp.kv_pool[s])[:, :512].astype(np.float64).mean(axis=0)
        if not (np.allclose(out[t], mean, atol=1e-12) and abs(lse[t] - np.log(len(s))) < 1e-12):
            failed.append("zero_query")
            break
    # Chain tree == causal attention (torch fp64).
    T, H, L = 5, 2, 7
    inp = make_inputs(batch=1, num_heads=H, prefix=[L], T=T, tree="chain", pool_slots=64,
                      nsplit=1, seed=44)
    out, _ = _run(lib, inp)
    kv = torch.from_numpy(bf16_bits_to_f32(inp.kv_pool[visible_slots(inp, 0, T - 1)])
                          .astype(np.float64))
    q = torch.from_numpy(bf16_bits_to_f32(inp.q).astype(np.float64)).permute(1, 0, 2)[None]
    mask = torch.ones(T, L + T, dtype=torch.bool)
    mask[:, L:] = torch.tril(torch.ones(T, T, dtype=torch.bool))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, kv[None, None].expand(1, H, L + T, 576), kv[None, None, :, :512].expand(1, H, L + T, 512),
        attn_mask=mask, scale=inp.softmax_scale)[0]
    got = torch.from_numpy(out.reshape(T, H, 512)).permute(1, 0, 2)
    if not torch.allclose(got, ref, rtol=0, atol=1e-12):
        failed.append("chain_causal")
    return failed


def test_unmutated_oracle_passes_battery(tmp_path):
    assert _battery(_compile(SRC, tmp_path, "clean")) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    failed = _battery(_compile(SRC.replace(old, new), tmp_path, name))
    assert failed, f"planted mistake {name} passed every pin"
