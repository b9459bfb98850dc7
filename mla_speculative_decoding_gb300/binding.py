"""Thin ctypes binding of libmlaverify.so (include/mla_verify.h).

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of the library. The functions keep the C names; tensors are torch
CUDA tensors (PyTorch provides device memory and streams), sizes are
taken from their shapes, and a non-zero C status raises MlaError. If the
library has not been built the import of a function fails loudly; there is
no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE_TOO_SMALL = -3
MLA_ERR_CUDA = -4
MLA_ERR_NOT_INITIALIZED = -5

MLA_STATUS_BAD_SLOT = 0x1
MLA_STATUS_BAD_PARENT = 0x2
MLA_STATUS_BAD_INDPTR = 0x4
MLA_STATUS_CAPACITY = 0x8
MLA_STATUS_BAD_PREFIX = 0x10
MLA_STATUS_EMPTY_ROW = 0x20
MLA_STATUS_TIMEOUT = 0x40

MLA_PARTIAL_PAIR = 0x4
MLA_PARTIAL_QUAD = 0x8
D_QK = 576
D_V = 512

_c_int = ctypes.c_int
_c_i64 = ctypes.c_int64
_c_size = ctypes.c_size_t
_c_f32 = ctypes.c_float
_vp = ctypes.c_void_p

_SIGS = {
    "mla_verify_status_string": (ctypes.c_char_p, [_c_int]),
    "mla_verify_version": (_c_int, []),
    "mla_verify_init": (_c_int, [_c_int]),
    "mla_verify_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "mla_verify_status_offset": (_c_size, []),
    "mla_verify_reset_status": (_c_int, [_vp, _vp]),
    "mla_build_verify_meta": (_c_int, [_vp, _c_i64, _c_i64, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                       _c_i64, _vp, _vp, _vp, _vp, _vp]),
    "mla_verify_attention": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp,
                                      _vp, _c_int, _c_int, _c_i64, _c_f32, _c_size, _vp]),
    "mla_verify_attention_anc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp,
                                          _vp, _c_int, _c_int, _c_i64, _c_f32, _c_size, _vp]),
    "mla_verify_attention_paged": (_c_int, [_vp, _vp, _vp, _c_i64, _c_i64, _vp, _vp, _vp, _vp,
                                            _c_int, _c_int, _vp, _vp, _vp, _c_int, _c_int, _c_i64,
                                            _c_f32, _c_size, _vp]),
    "mla_verify_partial_paged": (_c_int, [_vp, _vp, _vp, _c_i64, _c_i64, _vp, _vp, _vp, _vp,
                                          _c_int, _c_int, _vp, _c_int, _c_int, _c_i64, _c_f32,
                                          _c_size, _vp]),
    "mla_verify_partial": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _vp,
                                    _c_int, _c_int, _c_i64, _c_f32, _c_size, ctypes.c_uint, _vp]),
    "mla_verify_combine": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _c_size,
                                    _vp]),
    "mla_verify_noalloc_scratch_bytes": (_c_size, []),
    "mla_verify_attention_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _vp,
                                              _vp, _c_int, _c_int, _c_i64, _c_f32, _vp, _vp]),
    # include/mla_decode_steps.h
    "mla_tree_accept": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp,
                                 _vp]),
    "mla_kv_relocate": (_c_int, [_vp, _c_i64, _vp, _c_i64, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                 _vp, _vp]),
    "mla_fp8_indexer_logits": (_c_int, [_vp, _vp, _vp, _c_i64, _vp, _vp, _c_int, _c_int, _c_int,
                                        _vp, _vp, _vp]),
}

_LIB = None


class MlaError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmlaverify.so (building it in-tree first if it is missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing and not _build.up_to_date():
        _build.build_library()
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libmlaverify.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _LIB = lib
    return lib


def _check(fn, code):
    if code != MLA_OK:
        raise MlaError(fn, code)


def status_string(code: int) -> str:
    return load().mla_verify_status_string(int(code)).decode()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _p(t):
    """Device pointer of a torch tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _want(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")


def mla_verify_version() -> int:
    return int(load().mla_verify_version())


def mla_verify_init(device: int = None) -> None:
    if device is None:
        device = torch.cuda.current_device()
    _check("mla_verify_init", load().mla_verify_init(int(device)))


def mla_verify_workspace_bytes(batch: int, T: int, num_heads: int, nsplit: int) -> int:
    return int(load().mla_verify_workspace_bytes(batch, T, num_heads, nsplit))


def mla_verify_status_offset() -> int:
    return int(load().mla_verify_status_offset())


def alloc_workspace(batch, T, num_heads, nsplit, device="cuda"):
    n = mla_verify_workspace_bytes(batch, T, num_heads, nsplit)
    if n == 0:
        raise ValueError("shape outside the library's limits")
    return torch.empty(n, dtype=torch.uint8, device=device)


def status_word(workspace: torch.Tensor) -> torch.Tensor:
    """int32 view of the device status word inside a workspace."""
    off = mla_verify_status_offset()
    return workspace[off:off + 4].view(torch.int32)


def mla_verify_reset_status(status: torch.Tensor, stream=None) -> None:
    _check("mla_verify_reset_status", load().mla_verify_reset_status(_p(status), _stream(stream)))


def mla_build_verify_meta(req_to_token, req_pool_indices, prefix_lens, out_cache_loc, tree_parent,
                          kv_indptr, kv_indices, anc_mask, status, stream=None) -> None:
    """Device index/mask builder; capacity = kv_indices.numel()."""
    for t, n in ((req_to_token, "req_to_token"), (req_pool_indices, "req_pool_indices"),
                 (prefix_lens, "prefix_lens"), (out_cache_loc, "out_cache_loc"),
                 (tree_parent, "tree_parent"), (kv_indptr, "kv_indptr"),
                 (kv_indices, "kv_indices"), (status, "status")):
        _want(t, torch.int32, n)
    _want(anc_mask, torch.int64, "anc_mask")  # uint64 bits held in an int64 tensor
    B, T = tree_parent.shape
    rc = load().mla_build_verify_meta(
        _p(req_to_token), req_to_token.shape[1], req_to_token.shape[0], _p(req_pool_indices),
        _p(prefix_lens), _p(out_cache_loc), _p(tree_parent), B, T, kv_indices.numel(),
        _p(kv_indptr), _p(kv_indices), _p(anc_mask), _p(status), _stream(stream))
    _check("mla_build_verify_meta", rc)


def _attn_shapes(q, kv_pool, T, out, lse):
    _want(q, torch.bfloat16, "q")
    _want(kv_pool, torch.bfloat16, "kv_pool")
    if q.dim() != 3 or q.shape[2] != D_QK or q.shape[0] % T:
        raise ValueError("q must be [batch*T, H, 576]")
    if kv_pool.dim() != 2 or kv_pool.shape[1] != D_QK:
        raise ValueError("kv_pool must be [pool_slots, 576]")
    batch, H = q.shape[0] // T, q.shape[1]
    if out is not None:
        _want(out, torch.bfloat16, "out")
        if tuple(out.shape) != (batch * T, H, D_V):
            raise ValueError("out must be [batch*T, H, 512]")
    if lse is not None:
        _want(lse, torch.float32, "lse")
        if tuple(lse.shape) != (batch * T, H):
            raise ValueError("lse must be [batch*T, H]")
    return batch, H


def mla_verify_attention(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, T, nsplit,
                         workspace, out, lse, softmax_scale, stream=None) -> None:
    batch, H = _attn_shapes(q, kv_pool, T, out, lse)
    rc = load().mla_verify_attention(
        _p(q), _p(kv_pool), _p(kv_indices), _p(kv_indptr), _p(prefix_lens), _p(tree_parent), T,
        nsplit, _p(workspace), _p(out), _p(lse), batch, H, kv_pool.shape[0], float(softmax_scale),
        workspace.numel(), _stream(stream))
    _check("mla_verify_attention", rc)


def mla_verify_attention_anc(q, kv_pool, kv_indices, kv_indptr, prefix_lens, anc_mask, T, nsplit,
                             workspace, out, lse, softmax_scale, stream=None) -> None:
    batch, H = _attn_shapes(q, kv_pool, T, out, lse)
    rc = load().mla_verify_attention_anc(
        _p(q), _p(kv_pool), _p(kv_indices), _p(kv_indptr), _p(prefix_lens), _p(anc_mask), T,
        nsplit, _p(workspace), _p(out), _p(lse), batch, H, kv_pool.shape[0], float(softmax_scale),
        workspace.numel(), _stream(stream))
    _check("mla_verify_attention_anc", rc)


def mla_verify_attention_paged(q, kv_pool, req_to_token, req_pool_indices, prefix_lens,
                               out_cache_loc, tree_parent, T, nsplit, workspace, out, lse,
                               softmax_scale, stream=None) -> None:
    """Verify attention reading the page table directly (no built index list)."""
    batch, H = _attn_shapes(q, kv_pool, T, out, lse)
    rc = load().mla_verify_attention_paged(
        _p(q), _p(kv_pool), _p(req_to_token), req_to_token.shape[1], req_to_token.shape[0],
        _p(req_pool_indices), _p(prefix_lens), _p(out_cache_loc), _p(tree_parent), T, nsplit,
        _p(workspace), _p(out), _p(lse), batch, H, kv_pool.shape[0], float(softmax_scale),
        workspace.numel(), _stream(stream))
    _check("mla_verify_attention_paged", rc)


class BoundCall:
    """One C-ABI call with its arguments marshalled once (device pointers,
    sizes, scale and stream held as ctypes values); calling it issues the
    same call again. The tensors it was bound to must stay alive and keep
    their addresses (fixed buffers, as in a captured graph)."""

    def __init__(self, name, args, keep):
        self._name = name
        self._fn = getattr(load(), name)
        self._args = args
        self._keep = keep  # the tensors whose pointers the arguments hold

    def __call__(self) -> None:
        rc = self._fn(*self._args)
        if rc != MLA_OK:
            raise MlaError(self._name, rc)


def bind_verify_attention_paged(q, kv_pool, req_to_token, req_pool_indices, prefix_lens,
                                out_cache_loc, tree_parent, T, nsplit, workspace, out, lse,
                                softmax_scale, stream=None) -> BoundCall:
    """mla_verify_attention_paged with its arguments checked and marshalled
    once, for a caller that repeats the same call on fixed buffers."""
    batch, H = _attn_shapes(q, kv_pool, T, out, lse)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    args = (vp(_p(q)), vp(_p(kv_pool)), vp(_p(req_to_token)), i64(req_to_token.shape[1]),
            i64(req_to_token.shape[0]), vp(_p(req_pool_indices)), vp(_p(prefix_lens)),
            vp(_p(out_cache_loc)), vp(_p(tree_parent)), i32(T), i32(nsplit), vp(_p(workspace)),
            vp(_p(out)), vp(_p(lse)), i32(batch), i32(H), i64(kv_pool.shape[0]),
            ctypes.c_float(float(softmax_scale)), ctypes.c_size_t(workspace.numel()),
            vp(_stream(stream)))
    keep = (q, kv_pool, req_to_token, req_pool_indices, prefix_lens, out_cache_loc, tree_parent,
            workspace, out, lse)
    return BoundCall("mla_verify_attention_paged", args, keep)


def mla_verify_partial_paged(q, kv_pool, req_to_token, req_pool_indices, prefix_lens,
                             out_cache_loc, tree_parent, T, nsplit, workspace, softmax_scale,
                             stream=None) -> None:
    """The partial half of mla_verify_attention_paged."""
    batch, H = _attn_shapes(q, kv_pool, T, None, None)
    rc = load().mla_verify_partial_paged(
        _p(q), _p(kv_pool), _p(req_to_token), req_to_token.shape[1], req_to_token.shape[0],
        _p(req_pool_indices), _p(prefix_lens), _p(out_cache_loc), _p(tree_parent), T, nsplit,
        _p(workspace), batch, H, kv_pool.shape[0], float(softmax_scale), workspace.numel(),
        _stream(stream))
    _check("mla_verify_partial_paged", rc)


def mla_verify_partial(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, anc_mask, T,
                       nsplit, workspace, softmax_scale, flags=0, stream=None) -> None:
    batch, H = _attn_shapes(q, kv_pool, T, None, None)
    rc = load().mla_verify_partial(
        _p(q), _p(kv_pool), _p(kv_indices), _p(kv_indptr), _p(prefix_lens), _p(tree_parent),
        _p(anc_mask), T, nsplit, _p(workspace), batch, H, kv_pool.shape[0], float(softmax_scale),
        workspace.numel(), int(flags), _stream(stream))
    _check("mla_verify_partial", rc)


def mla_verify_combine(workspace, batch, T, num_heads, nsplit, out, lse, stream=None) -> None:
    rc = load().mla_verify_combine(_p(workspace), batch, T, num_heads, nsplit, _p(out), _p(lse),
                                   workspace.numel(), _stream(stream))
    _check("mla_verify_combine", rc)


def partials(workspace, batch, T, num_heads, nsplit):
    """Views (lse_part [rows, nsplit], o_part [rows, nsplit, 512]) into a workspace."""
    rows = batch * T * num_heads
    n = rows * nsplit
    lse_off = 256
    o_off = lse_off + ((n * 4 + 255) // 256) * 256
    lse_part = workspace[lse_off:lse_off + n * 4].view(torch.float32).view(rows, nsplit)
    o_part = workspace[o_off:o_off + n * 512 * 4].view(torch.float32).view(rows, nsplit, 512)
    return lse_part, o_part


def mla_verify_noalloc_scratch_bytes() -> int:
    return int(load().mla_verify_noalloc_scratch_bytes())


def mla_verify_attention_noalloc(q, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent, T,
                                 nsplit, out, lse, softmax_scale, status=None,
                                 stream=None) -> None:
    """Verify call without a workspace: the partials use the library's fixed
    device scratch area (for callers that cannot allocate device memory)."""
    batch, H = _attn_shapes(q, kv_pool, T, out, lse)
    _want(status, torch.int32, "status")
    rc = load().mla_verify_attention_noalloc(
        _p(q), _p(kv_pool), _p(kv_indices), _p(kv_indptr), _p(prefix_lens), _p(tree_parent), T,
        nsplit, _p(out), _p(lse), batch, H, kv_pool.shape[0], float(softmax_scale), _p(status),
        _stream(stream))
    _check("mla_verify_attention_noalloc", rc)



# ---------------------------------------------------------------- decode steps (mla_decode_steps.h)
def mla_tree_accept(tree_parent, draft_tokens, target_argmax, out_cache_loc, commit_len,
                    accepted_nodes, kept_slots, next_tokens, status, stream=None) -> None:
    """Greedy acceptance along each request's draft tree; all int32 CUDA
    tensors, [B, T] inputs and outputs, commit_len [B]."""
    for name, t in (("tree_parent", tree_parent), ("draft_tokens", draft_tokens),
                    ("target_argmax", target_argmax), ("out_cache_loc", out_cache_loc),
                    ("commit_len", commit_len), ("accepted_nodes", accepted_nodes),
                    ("kept_slots", kept_slots), ("next_tokens", next_tokens), ("status", status)):
        _want(t, torch.int32, name)
    B, T = tree_parent.shape
    rc = load().mla_tree_accept(_p(tree_parent), _p(draft_tokens), _p(target_argmax),
                                _p(out_cache_loc), B, T, _p(commit_len), _p(accepted_nodes),
                                _p(kept_slots), _p(next_tokens), _p(status), _stream(stream))
    _check("mla_tree_accept", rc)


def mla_kv_relocate(kv_pool, req_to_token, req_pool_indices, prefix_lens, dst_start, progress,
                    budget, status, stream=None) -> None:
    """One relocation call (moves up to `budget` rows per request)."""
    _want(kv_pool, torch.bfloat16, "kv_pool")
    for name, t in (("req_to_token", req_to_token), ("req_pool_indices", req_pool_indices),
                    ("prefix_lens", prefix_lens), ("dst_start", dst_start),
                    ("progress", progress), ("status", status)):
        _want(t, torch.int32, name)
    rc = load().mla_kv_relocate(_p(kv_pool), kv_pool.shape[0], _p(req_to_token),
                                req_to_token.shape[1], _p(req_pool_indices), _p(prefix_lens),
                                _p(dst_start), _p(progress), prefix_lens.shape[0], int(budget),
                                _p(status), _stream(stream))
    _check("mla_kv_relocate", rc)


def mla_fp8_indexer_logits(q, weights, kv_blocks, block_table, seq_lens, logits, status,
                           stream=None) -> None:
    """Indexer logits [B, max_pages * 64] (fp32) from fp8-e4m3 bytes q
    [B, H, 128] (uint8), weights [B, H] fp32, kv_blocks [nblocks, 8448] uint8,
    block_table [B, max_pages] int32, seq_lens [B] int32."""
    _want(q, torch.uint8, "q")
    _want(kv_blocks, torch.uint8, "kv_blocks")
    _want(weights, torch.float32, "weights")
    _want(logits, torch.float32, "logits")
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens), ("status", status)):
        _want(t, torch.int32, name)
    B, H, _ = q.shape
    rc = load().mla_fp8_indexer_logits(_p(q), _p(weights), _p(kv_blocks), kv_blocks.shape[0],
                                       _p(block_table), _p(seq_lens), B, H, block_table.shape[1],
                                       _p(logits), _p(status), _stream(stream))
    _check("mla_fp8_indexer_logits", rc)
