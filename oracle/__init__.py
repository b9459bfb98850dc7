"""CPU fp64 oracle for MLA tree-verify attention.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference leg may import this package. The CUDA product path
never imports, links or runs it, and the two share no code: the only thing
both sides consume is the seeded input generator in `workloads`.

Functions:
  build_meta(inp)                -> (kv_indptr, kv_indices, anc)   exact ints
  verify_attention(inp, indptr, indices, rows=None) -> (out f64 [n,512], lse f64 [n])
  tree_accept(parent, draft, target, loc) -> (commit_len, accepted_nodes, kept_slots, next_tokens)
  kv_relocate(state, budget)     -> relocated copy of (kv_pool, req_to_token, progress)
  fp8_indexer_logits(ix)         -> logits f64 [B, max_pages * 64]
  e4m3_value(code)               -> the fp8 (e4m3) value of a byte
(the last four in next_rows_oracle.c).

The arithmetic lives in mla_verify_oracle.c (plain loops, fp64), which
cites the page passages it follows. Every function has pins in
tests/test_oracle_*.py (brute force, a library special case, closed forms
and invariants).
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None
_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)

ERRORS = {-1: "bad argument", -2: "invalid tree", -3: "bad index", -4: "out of memory"}


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_build_meta.argtypes = [_i32p, ctypes.c_int64, _i32p, _i32p, _i32p, _i32p,
                                          ctypes.c_int, ctypes.c_int, _i32p, _i32p, _u64p]
        lib.oracle_build_meta.restype = ctypes.c_int
        lib.oracle_verify_attention.argtypes = [_u16p, _u16p, ctypes.c_int64, _i32p, _i32p,
                                                _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_double, _i64p,
                                                ctypes.c_int64, _f64p, _f64p, ctypes.c_int]
        lib.oracle_verify_attention.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_tree_accept.argtypes = [_i32p] * 4 + [ctypes.c_int] * 2 + [_i32p] * 4
        lib.oracle_tree_accept.restype = ctypes.c_int
        lib.oracle_kv_relocate.argtypes = [_u16p, ctypes.c_int64, _i32p, ctypes.c_int64, _i32p,
                                           _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int]
        lib.oracle_kv_relocate.restype = ctypes.c_int
        lib.oracle_fp8_indexer_logits.argtypes = [
            ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_float),
            ctypes.POINTER(ctypes.c_uint8), ctypes.c_int64, _i32p, _i32p, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, _f64p]
        lib.oracle_fp8_indexer_logits.restype = ctypes.c_int
        lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        _LIB = lib
    return _LIB


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def build_meta(inp, tree_parent=None):
    """Combined KV index list, its offsets, and ancestor-or-self bit sets."""
    T, B = inp.T, inp.batch
    par = _c(inp.tree_parent if tree_parent is None else tree_parent, np.int32)
    L = _c(inp.prefix_lens, np.int32)
    indptr = np.zeros(B + 1, dtype=np.int32)
    n = int(L.astype(np.int64).sum() + B * T)
    indices = np.zeros(max(n, 1), dtype=np.int32)
    anc = np.zeros(B * T, dtype=np.uint64)
    r2t = _c(inp.req_to_token, np.int32)
    rc = _lib().oracle_build_meta(_ptr(r2t, _i32p), r2t.shape[1],
                                  _ptr(_c(inp.req_pool_indices, np.int32), _i32p),
                                  _ptr(L, _i32p), _ptr(_c(inp.out_cache_loc, np.int32), _i32p),
                                  _ptr(par, _i32p), B, T, _ptr(indptr, _i32p),
                                  _ptr(indices, _i32p), _ptr(anc, _u64p))
    if rc != 0:
        raise ValueError(f"oracle_build_meta: {ERRORS.get(rc, rc)}")
    return indptr, indices[:n], anc.reshape(B, T)


def verify_attention(inp, kv_indptr, kv_indices, rows=None, nthreads=0, tree_parent=None,
                     q=None, prefix_lens=None):
    """fp64 reference output rows and their log-sum-exp.

    rows: optional iterable of row ids n = (b*T + t)*H + h; default all rows.
    Returns (out [len(rows), 512] float64, lse [len(rows)] float64).
    """
    q = _c(inp.q if q is None else q, np.uint16)
    kv = inp.kv_pool
    if not kv.flags.c_contiguous:
        kv = np.ascontiguousarray(kv)
    par = _c(inp.tree_parent if tree_parent is None else tree_parent, np.int32)
    L = _c(inp.prefix_lens if prefix_lens is None else prefix_lens, np.int32)
    indptr = _c(kv_indptr, np.int32)
    indices = _c(kv_indices, np.int32)
    if indices.size == 0:
        indices = np.zeros(1, dtype=np.int32)
    if rows is None:
        nrows = inp.num_rows
        rows_arr = None
    else:
        rows_arr = _c(np.asarray(list(rows) if not isinstance(rows, np.ndarray) else rows),
                      np.int64)
        nrows = rows_arr.size
    out = np.zeros((max(nrows, 1), 512), dtype=np.float64)
    lse = np.zeros(max(nrows, 1), dtype=np.float64)
    rc = _lib().oracle_verify_attention(
        _ptr(q, _u16p), _ptr(kv, _u16p), kv.shape[0], _ptr(indices, _i32p), _ptr(indptr, _i32p),
        _ptr(L, _i32p), _ptr(par, _i32p), inp.batch, inp.T, inp.num_heads,
        float(inp.softmax_scale), None if rows_arr is None else _ptr(rows_arr, _i64p), nrows,
        _ptr(out, _f64p), _ptr(lse, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_verify_attention: {ERRORS.get(rc, rc)}")
    return out[:nrows], lse[:nrows]


def row_id(inp, b, t, h):
    return (b * inp.T + t) * inp.num_heads + h


class OracleError(RuntimeError):
    pass


def tree_accept(parent, draft, target, loc):
    """Greedy acceptance along each request's draft tree ([B, T] int32 inputs).
    Returns (commit_len [B], accepted_nodes [B, T], kept_slots [B, T],
    next_tokens [B, T]), padded with -1."""
    parent = _c(parent, np.int32)
    draft = _c(draft, np.int32)
    target = _c(target, np.int32)
    loc = _c(loc, np.int32)
    B, T = parent.shape
    commit = np.zeros(B, np.int32)
    an = np.zeros((B, T), np.int32)
    ks = np.zeros((B, T), np.int32)
    nt = np.zeros((B, T), np.int32)
    rc = _lib().oracle_tree_accept(_ptr(parent, _i32p), _ptr(draft, _i32p), _ptr(target, _i32p),
                                   _ptr(loc, _i32p), B, T, _ptr(commit, _i32p), _ptr(an, _i32p),
                                   _ptr(ks, _i32p), _ptr(nt, _i32p))
    if rc != 0:
        raise OracleError(f"tree_accept: {ERRORS.get(rc, rc)}")
    return commit, an, ks, nt


def kv_relocate(kv_pool, req_to_token, req_pool_indices, prefix_lens, dst_start, progress, budget):
    """One relocation call on copies of the state; returns the new
    (kv_pool, req_to_token, progress). Raises on a contract violation
    (-5: a destination slot is live or targeted twice)."""
    pool = np.array(kv_pool, dtype=np.uint16, copy=True, order="C")
    r2t = np.array(req_to_token, dtype=np.int32, copy=True, order="C")
    prog = np.array(progress, dtype=np.int32, copy=True)
    rpi = _c(req_pool_indices, np.int32)
    L = _c(prefix_lens, np.int32)
    dst = _c(dst_start, np.int32)
    rc = _lib().oracle_kv_relocate(_ptr(pool, _u16p), pool.shape[0], _ptr(r2t, _i32p),
                                   r2t.shape[1], _ptr(rpi, _i32p), _ptr(L, _i32p),
                                   _ptr(dst, _i32p), _ptr(prog, _i32p), len(L), int(budget))
    if rc != 0:
        raise OracleError(f"kv_relocate: {ERRORS.get(rc, 'destination slot live or shared' if rc == -5 else rc)}")
    return pool, r2t, prog


def fp8_indexer_logits(q, weights, kv_blocks, block_table, seq_lens):
    """Indexer logits [B, max_pages * 64] (fp64) from fp8 bytes q [B, H, 128],
    fp32 weights [B, H], 8448-byte KV blocks [nblocks, 8448], block_table
    [B, max_pages], seq_lens [B]."""
    q = _c(q, np.uint8)
    w = _c(weights, np.float32)
    kv = _c(kv_blocks, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H, _ = q.shape
    P = bt.shape[1]
    out = np.zeros((B, P * 64), np.float64)
    rc = _lib().oracle_fp8_indexer_logits(
        q.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), w.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
        kv.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), kv.shape[0], _ptr(bt, _i32p),
        _ptr(sl, _i32p), B, H, P, _ptr(out, _f64p))
    if rc != 0:
        raise OracleError(f"fp8_indexer_logits: {ERRORS.get(rc, rc)}")
    return out


def e4m3_value(code):
    return _lib().oracle_e4m3_value(int(code))
