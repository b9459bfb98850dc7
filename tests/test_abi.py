"""The C-ABI library builds, loads, and exports every symbol its header
declares; host-side logic (workspace sizing, argument checks) behaves as
documented. No compute call is made here (no GPU needed)."""

import ctypes
import glob
import json
import os
import re
import subprocess

import pytest

import mla_speculative_decoding_gb300 as mv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def _declared():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return mv.load()


def test_exports_match_header(lib):
    declared = _declared()
    assert len(declared) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", mv.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines()
                       if ln.split() and ln.split()[-1].startswith("mla_")})
    assert exported == declared
    for name in declared:
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert mv.mla_verify_version() == 100
    assert mv.status_string(0) == "MLA_OK"
    assert mv.status_string(-3) == "MLA_ERR_WORKSPACE_TOO_SMALL"
    assert mv.status_string(-99) == "MLA_ERR_UNKNOWN"


def test_workspace_bytes_follow_partial_count(lib):
    """One partial (512 fp32 + one fp32 lse) per (request, token, head, split):
    the pages' grid arithmetic 1 x 9 x 8 x 16 = 1152 partials."""
    fig = json.load(open(os.path.join(ROOT, "tests", "golden", "page_figures.json")))
    g = fig["partials_grid"]
    for ns, parts in ((g["nsplit_before"], g["blocks_before"]), (g["nsplit_after"], g["blocks_after"])):
        n = mv.mla_verify_workspace_bytes(g["batch"], g["tree_tokens"], g["heads"], ns)
        lse_bytes = (parts * 4 + 255) // 256 * 256
        assert n == 256 + lse_bytes + parts * 512 * 4
    assert mv.mla_verify_status_offset() == 0


@pytest.mark.parametrize("args", [(0, 4, 8, 4), (1, 0, 8, 4), (1, 65, 8, 4), (1, 4, 0, 4),
                                  (1, 4, 129, 4), (1, 4, 8, 0), (1, 4, 8, 129), (65536, 1, 1, 1)])
def test_workspace_bytes_rejects_out_of_limits(lib, args):
    assert mv.mla_verify_workspace_bytes(*args) == 0


def test_limits_accept_maximum_sizes(lib):
    assert mv.mla_verify_workspace_bytes(1, 64, 128, 128) > 0


def _vp(x):
    return ctypes.c_void_p(x)


def test_attention_argument_checks_before_any_launch(lib):
    """Invalid host-side arguments return an error code before any CUDA call."""
    A = 0x10000  # aligned, never dereferenced: every call below fails its checks first
    ws_need = mv.mla_verify_workspace_bytes(1, 4, 8, 4)
    f = lib.mla_verify_attention
    ok = dict(q=A, kv=A, idx=A, ptr=A, pl=A, par=A, T=4, ns=4, ws=A, out=A, lse=A, B=1, H=8,
              slots=4096, scale=0.07, wsb=ws_need)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(_vp(a["q"]), _vp(a["kv"]), _vp(a["idx"]), _vp(a["ptr"]), _vp(a["pl"]),
                 _vp(a["par"]), a["T"], a["ns"], _vp(a["ws"]), _vp(a["out"]), _vp(a["lse"]),
                 a["B"], a["H"], a["slots"], a["scale"], a["wsb"], None)

    assert call(q=0) == -1
    assert call(par=0) == -1
    assert call(q=A + 2) == -1            # q not 16-byte aligned
    assert call(ws=A + 64) == -1          # workspace not 256-byte aligned
    assert call(T=65) == -1
    assert call(ns=0) == -1
    assert call(H=129) == -1
    assert call(scale=0.0) == -1
    assert call(scale=float("inf")) == -1
    assert call(slots=0) == -1
    assert call(wsb=ws_need - 1) == -3
    # Partial: exactly one mask source.
    g = lib.mla_verify_partial
    assert g(_vp(A), _vp(A), _vp(A), _vp(A), _vp(A), _vp(A), _vp(A), 4, 4, _vp(A), 1, 8, 4096,
             0.07, ws_need, 0, None) == -1
    assert g(_vp(A), _vp(A), _vp(A), _vp(A), _vp(A), None, None, 4, 4, _vp(A), 1, 8, 4096,
             0.07, ws_need, 0, None) == -1


def test_builder_argument_checks(lib):
    A = 0x10000
    f = lib.mla_build_verify_meta
    base = [_vp(A), 100, 2, _vp(A), _vp(A), _vp(A), _vp(A), 1, 4, 1000, _vp(A), _vp(A), _vp(A),
            _vp(A), None]
    for i, bad in [(0, _vp(0)), (7, 0), (8, 65), (1, 0), (2, 0), (9, 0), (9, 2 ** 31), (13, _vp(0))]:
        a = list(base)
        a[i] = bad
        assert f(*a) == -1, i
