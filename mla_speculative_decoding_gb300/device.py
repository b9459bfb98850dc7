"""Device-side buffers for one verify shape (PyTorch used for memory only).

DeviceInputs holds the inputs of a verify call as CUDA tensors (bf16 data
is carried as raw bits and viewed as torch.bfloat16). `step()` runs the
whole verify path through the C ABI: the index/mask builder, the split-KV
partial kernel and the combine, all on one stream, with fixed buffers (so
it can be captured in a CUDA graph).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import binding as B


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _i32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


@dataclass
class DeviceInputs:
    batch: int
    T: int
    num_heads: int
    nsplit: int
    softmax_scale: float
    q: torch.Tensor               # bf16 [B*T, H, 576]
    kv_pool: torch.Tensor         # bf16 [slots, 576]
    req_to_token: torch.Tensor    # int32 [R, stride]
    req_pool_indices: torch.Tensor
    prefix_lens: torch.Tensor
    out_cache_loc: torch.Tensor
    tree_parent: torch.Tensor     # int32 [B, T]
    capacity: int
    # outputs and fixed scratch
    kv_indptr: torch.Tensor = None
    kv_indices: torch.Tensor = None
    anc_mask: torch.Tensor = None
    workspace: torch.Tensor = None
    out: torch.Tensor = None
    lse: torch.Tensor = None
    # One byte buffer each for the per-step inputs (q, tree_parent,
    # prefix_lens, req_pool_indices, out_cache_loc) and outputs (out, lse);
    # the named tensors are views into them, so a step's host data moves in
    # one copy each way.
    step_in: torch.Tensor = None
    step_out: torch.Tensor = None

    STEP_INPUTS = ("q", "tree_parent", "prefix_lens", "req_pool_indices", "out_cache_loc")

    def allocate(self):
        dev = self.q.device
        self.kv_indptr = torch.zeros(self.batch + 1, dtype=torch.int32, device=dev)
        self.kv_indices = torch.zeros(max(self.capacity, 1), dtype=torch.int32, device=dev)
        self.anc_mask = torch.zeros(self.batch * self.T, dtype=torch.int64, device=dev)
        self.workspace = B.alloc_workspace(self.batch, self.T, self.num_heads, self.nsplit, dev)
        self.workspace[:256].zero_()
        self.step_in = _pack(self, self.STEP_INPUTS, dev)
        out = torch.empty(self.batch * self.T, self.num_heads, B.D_V, dtype=torch.bfloat16,
                          device=dev)
        lse = torch.empty(self.batch * self.T, self.num_heads, dtype=torch.float32, device=dev)
        self.out, self.lse = out, lse
        self.step_out = _pack(self, ("out", "lse"), dev)
        return self

    @property
    def status(self) -> torch.Tensor:
        return B.status_word(self.workspace)

    def build(self, stream=None):
        B.mla_build_verify_meta(self.req_to_token, self.req_pool_indices, self.prefix_lens,
                                self.out_cache_loc, self.tree_parent, self.kv_indptr,
                                self.kv_indices, self.anc_mask, self.status, stream)

    def attention(self, use_anc=True, stream=None):
        if use_anc:
            B.mla_verify_attention_anc(self.q, self.kv_pool, self.kv_indices, self.kv_indptr,
                                       self.prefix_lens, self.anc_mask, self.T, self.nsplit,
                                       self.workspace, self.out, self.lse, self.softmax_scale,
                                       stream)
        else:
            B.mla_verify_attention(self.q, self.kv_pool, self.kv_indices, self.kv_indptr,
                                   self.prefix_lens, self.tree_parent, self.T, self.nsplit,
                                   self.workspace, self.out, self.lse, self.softmax_scale, stream)

    def partial(self, flags=0, use_anc=True, stream=None):
        B.mla_verify_partial(self.q, self.kv_pool, self.kv_indices, self.kv_indptr,
                             self.prefix_lens, None if use_anc else self.tree_parent,
                             self.anc_mask if use_anc else None, self.T, self.nsplit,
                             self.workspace, self.softmax_scale, flags, stream)

    def combine(self, stream=None):
        B.mla_verify_combine(self.workspace, self.batch, self.T, self.num_heads, self.nsplit,
                             self.out, self.lse, stream)

    def step(self, stream=None):
        """One pass of the whole verify path: build, partial, combine."""
        self.build(stream)
        self.attention(True, stream)

    def step_paged(self, stream=None):
        """The same pass with the index build fused into the partial kernels'
        gathers (they read the page table): partial, combine."""
        B.mla_verify_attention_paged(self.q, self.kv_pool, self.req_to_token, self.req_pool_indices,
                                     self.prefix_lens, self.out_cache_loc, self.tree_parent, self.T,
                                     self.nsplit, self.workspace, self.out, self.lse,
                                     self.softmax_scale, stream)

    def bound_step_paged(self, stream=None) -> B.BoundCall:
        """step_paged with its arguments marshalled once (for a loop that
        repeats the call on these fixed buffers)."""
        return B.bind_verify_attention_paged(
            self.q, self.kv_pool, self.req_to_token, self.req_pool_indices, self.prefix_lens,
            self.out_cache_loc, self.tree_parent, self.T, self.nsplit, self.workspace, self.out,
            self.lse, self.softmax_scale, stream)

    def partial_paged(self, stream=None):
        """The partial half of step_paged (combine() finishes it)."""
        B.mla_verify_partial_paged(self.q, self.kv_pool, self.req_to_token, self.req_pool_indices,
                                   self.prefix_lens, self.out_cache_loc, self.tree_parent, self.T,
                                   self.nsplit, self.workspace, self.softmax_scale, stream)


def _pack(d: DeviceInputs, names, dev) -> torch.Tensor:
    """Moves the named tensors of `d` into one byte buffer (each at a 256-byte
    aligned offset) and rebinds the names to views of it; returns the buffer."""
    offs, total = [], 0
    for n in names:
        t = getattr(d, n)
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    for n, off in zip(names, offs):
        t = getattr(d, n)
        nb = t.numel() * t.element_size()
        v = buf[off:off + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        setattr(d, n, v)
    return buf


def to_device(inp, device="cuda", nsplit=None, capacity=None) -> DeviceInputs:
    """Copy a host-side verify workload (numpy arrays) to the device."""
    stride = inp.req_to_token.shape[1]
    cap = capacity if capacity is not None else inp.batch * (stride + inp.T)
    d = DeviceInputs(
        batch=inp.batch, T=inp.T, num_heads=inp.num_heads,
        nsplit=inp.nsplit if nsplit is None else nsplit, softmax_scale=inp.softmax_scale,
        q=_bf16(inp.q, device), kv_pool=_bf16(inp.kv_pool, device),
        req_to_token=_i32(inp.req_to_token, device),
        req_pool_indices=_i32(inp.req_pool_indices, device),
        prefix_lens=_i32(inp.prefix_lens, device), out_cache_loc=_i32(inp.out_cache_loc, device),
        tree_parent=_i32(inp.tree_parent, device), capacity=int(cap))
    return d.allocate()
