"""Pins from figures the pages print (tests/golden/page_figures.json)."""

import json
import os

import numpy as np

import oracle
from workloads import D_QK, D_V, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
FIG = json.load(open(os.path.join(HERE, "golden", "page_figures.json")))


def test_latent_row_is_576_bf16():
    k = FIG["kv_row"]
    assert k["d_latent"] + k["d_rope"] == D_QK and k["d_latent"] == D_V
    row_bytes = D_QK * k["bytes_per_elem_bf16"]
    assert row_bytes == 1152
    # ~68 KB per token across 61 layers.
    assert abs(row_bytes * k["layers"] / 1024 - k["kb_per_token_all_layers_approx"]) < 1.0


def test_step_bytes_and_effective_bandwidth():
    s = FIG["kv_step_bytes"]
    gb = s["context"] * 1152 * s["layers"] / 1e9
    assert abs(gb - s["gb_per_step_approx"]) < 0.2
    gbps = gb / (s["step_ms"] / 1e3)
    assert abs(gbps - s["effective_gbps_approx"]) < 1.0


def test_partial_count_reading_of_nsplit():
    """NSPLIT multiplies the number of partial results: one partial per
    (request, tree token, head, split)."""
    g = FIG["partials_grid"]
    assert g["batch"] * g["tree_tokens"] * g["heads"] * g["nsplit_before"] == g["blocks_before"]
    assert g["batch"] * g["tree_tokens"] * g["heads"] * g["nsplit_after"] == g["blocks_after"]


def test_oracle_on_the_pages_parity_shape():
    """The shape the pages validated on (21 prefix + 9 draft tokens) runs through
    the oracle and its output rows are convex combinations of V rows."""
    p = FIG["parity_scale"]
    inp = make_inputs(batch=1, num_heads=8, prefix=[p["prefix"]], T=p["draft"], tree="random",
                      pool_slots=4096, nsplit=16, seed=5)
    ip, ix, _ = oracle.build_meta(inp)
    out, lse = oracle.verify_attention(inp, ip, ix)
    from workloads import bf16_bits_to_f32
    v = bf16_bits_to_f32(inp.kv_pool[ix])[:, :512].astype(np.float64)
    assert np.all(out <= v.max(axis=0) + 1e-12) and np.all(out >= v.min(axis=0) - 1e-12)
    assert np.all(np.isfinite(lse))
