"""Planted mistakes in the oracle of the steps beside the verify attention are
caught by their pins (tests/test_oracle_next_rows.py).

Each case copies next_rows_oracle.c, plants one plausible slip by text
substitution, compiles it with the unchanged verify oracle on the CPU, points
the oracle package at the copy and runs the pins for that function. The
untouched source must pass and every planted slip must fail."""

import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_next_rows as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "next_rows_oracle.c")).read()
VERIFY_SRC = os.path.join(ROOT, "oracle", "mla_verify_oracle.c")

ACCEPT = [pins.test_accept_chain_all_match, pins.test_accept_nothing_matches,
          pins.test_accept_repeated_sibling_token_takes_lowest_node,
          lambda: pins.test_accept_properties_random("random", 0.9)]
RELOC = [pins.test_relocation_keeps_attention_bitwise,
         pins.test_relocation_budget_progress_and_exact_copies,
         pins.test_relocation_in_place_rows_and_contract]
INDEX = [pins.test_e4m3_decoding_matches_torch_float8,
         lambda: pins.test_indexer_matches_torch_fp64([1, 64, 65, 200]),
         pins.test_indexer_page_table_indirection_invariance, pins.test_indexer_zero_query_and_relu]

MUTATIONS = {
    "accept_highest_child": ("nxt = c;\n                    break;", "nxt = c;", ACCEPT),
    "accept_no_bonus": ("nt[n] = tgt[cur];", "nt[n] = tok[cur];", ACCEPT),
    "accept_root_not_kept": ("ks[0] = loc[0];", "ks[0] = -1;", ACCEPT),
    "reloc_budget_short": ("if (s != d) memcpy", "if (s != d && j + 1 < j0 + n) memcpy", RELOC),
    "reloc_shifted_destination": ("const int64_t s = row[j], d = (int64_t)dst_start[b] + j;",
                                  "const int64_t s = row[j], d = (int64_t)dst_start[b] + j + 1;",
                                  RELOC),
    "reloc_table_not_rewritten": ("            row[j] = (int32_t)d;\n", "", RELOC),
    "index_no_relu": ("(dot > 0.0 ? dot : 0.0)", "dot", INDEX),
    "index_no_scale": ("*o = (double)sf * acc;", "*o = acc;", INDEX),
    "index_wrong_scale_slot": ("base + 8192 + 4 * i, 4);", "base + 8192 + 4 * (i ^ 1), 4);", INDEX),
    "e4m3_bias": ("x = ldexp(1.0 + (double)m / 8.0, e - 7);",
                  "x = ldexp(1.0 + (double)m / 8.0, e - 8);", INDEX),
    "index_last_position_dropped": ("if (pos >= len) {", "if (pos + 1 >= len) {", INDEX),
}


def _compile(src, tmp_path, name):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(c), VERIFY_SRC, "-o",
                    str(so), "-lm"], check=True, capture_output=True)
    return str(so)


def _with_lib(path, battery):
    """Run the battery with the oracle package bound to the library at path;
    returns True if every pin passes."""
    saved = oracle._LIB
    try:
        oracle._LIB = None
        real_build = oracle._build.build
        oracle._build.build = lambda *a, **k: path
        try:
            for pin in battery:
                try:
                    pin()
                except (AssertionError, oracle.OracleError):
                    return False
            return True
        finally:
            oracle._build.build = real_build
    finally:
        oracle._LIB = saved


def test_untouched_source_passes(tmp_path):
    so = _compile(SRC, tmp_path, "clean")
    assert _with_lib(so, ACCEPT + RELOC + INDEX)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new, battery = MUTATIONS[name]
    assert SRC.count(old) >= 1, f"mutation anchor for {name} not found"
    so = _compile(SRC.replace(old, new), tmp_path, name)
    assert not _with_lib(so, battery), f"planted mistake {name} was not caught"
