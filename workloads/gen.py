"""Seeded input generator for MLA tree-verify attention workloads.

Shapes follow the absorbed-latent MLA verify step described on the page
"The Custom sm_120 Verify Kernel: From 0.7 tok/s to 3-6x Decode Speedup on
Blackwell Consumer GPUs" (Parts I, VI, VII, IX): one 576-wide bf16 latent row
per token (512 latent + 64 RoPE dims), a page_size-1 KV pool whose slots are
scattered, per-request prefix slots held in a req_to_token table, and T draft
tree tokens whose slots come from out_cache_loc.

Draw order for one workload (numpy default_rng(seed)):
  1. prefix lengths L_b (only when drawn at random),
  2. tree parents (parent[0] = -1, parent[i] uniform in [0, i-1]),
  3. one permutation of the pool; its first n entries are the used slots
     (drawn for the contiguous placement too, so that both placements see
     the same later draws),
  4. q ~ N(0,1) float32, rounded to bf16 (round to nearest even),
  5. latent KV rows ~ N(0,1) float32 for the n used keys in logical order
     (request, then prefix position, then tree node), rounded to bf16.
Unused pool slots hold a bf16 NaN so that any stray read shows up.

Nothing here computes attention, softmax, visibility masks or the combined
KV index list.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D_QK = 576  # 512 latent + 64 RoPE dims per query head and per latent KV row
D_V = 512  # V is the first 512 dims of the latent row
BF16_NAN = np.uint16(0x7FC0)

# Five synthetic verify workloads. Seeds: the tiny one is fixed at 0; the
# others take 1..4.
CONFIGS = {
    1: dict(name="tiny", batch=1, num_heads=8, prefix="fixed:256", T=4, tree="chain",
            pool_slots=4096, nsplit=4, seed=0),
    2: dict(name="short", batch=1, num_heads=8, prefix="fixed:4096", T=16, tree="random",
            pool_slots=200_000, nsplit=64, seed=1),
    3: dict(name="mid", batch=1, num_heads=8, prefix="fixed:65536", T=16, tree="random",
            pool_slots=200_000, nsplit=64, seed=2),
    4: dict(name="long", batch=1, num_heads=8, prefix="fixed:184728", T=64, tree="random",
            pool_slots=195_011, nsplit=64, seed=3),
    5: dict(name="batched", batch=8, num_heads=64, prefix="uniform:1024:131072", T=16,
            tree="random", pool_slots=1_200_000, nsplit=64, seed=4),
}

# Sparse-MLA decode: each of 16 requests' 64 heads attend over a top-k list of
# 512 scattered slots (given as the request's prefix) plus the token's own
# slot (T = 1), split 8 ways over the keys.
SPARSE_DECODE = dict(name="sparse-decode", batch=16, num_heads=64, prefix="fixed:512", T=1,
                     tree="chain", pool_slots=1_200_000, nsplit=8, seed=5)


def f32_to_bf16_bits(x: np.ndarray, chunk: int = 1 << 24) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1).view(np.uint32)
    out = np.empty(flat.shape, dtype=np.uint16)
    for s in range(0, flat.size, chunk):
        b = flat[s:s + chunk].astype(np.uint64)
        b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
        out[s:s + chunk] = b.astype(np.uint16)
    return out.reshape(x.shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass
class VerifyInputs:
    """Host-side inputs of one verify call (all numpy, C-contiguous)."""

    name: str
    batch: int
    num_heads: int
    T: int
    prefix_lens: np.ndarray        # int32 [B]
    tree_parent: np.ndarray        # int32 [B, T]; parent[b, 0] = -1
    req_to_token: np.ndarray       # int32 [R, stride]; row r: token position -> pool slot
    req_pool_indices: np.ndarray   # int32 [B]; request b uses row req_pool_indices[b]
    out_cache_loc: np.ndarray      # int32 [B*T]; pool slot of each draft-tree token
    q: np.ndarray                  # uint16 (bf16 bits) [B*T, H, 576]
    kv_pool: np.ndarray            # uint16 (bf16 bits) [pool_slots, 576]
    nsplit: int
    softmax_scale: float
    seed: int
    placement: str
    meta: dict = field(default_factory=dict)

    @property
    def pool_slots(self) -> int:
        return int(self.kv_pool.shape[0])

    @property
    def total_keys(self) -> int:
        return int(self.prefix_lens.astype(np.int64).sum() + self.batch * self.T)

    @property
    def num_rows(self) -> int:
        return self.batch * self.T * self.num_heads


def _draw_prefix(rng, spec, batch):
    if isinstance(spec, (list, tuple, np.ndarray)):
        arr = np.asarray(spec, dtype=np.int64)
        if arr.size == 1 and batch > 1:
            arr = np.full(batch, int(arr[0]), dtype=np.int64)
        return arr
    kind, *args = spec.split(":")
    if kind == "fixed":
        return np.full(batch, int(args[0]), dtype=np.int64)
    if kind == "uniform":
        lo, hi = int(args[0]), int(args[1])
        return rng.integers(lo, hi, size=batch, endpoint=True).astype(np.int64)
    raise ValueError(f"unknown prefix spec {spec!r}")


def _draw_tree(rng, spec, batch, T):
    if isinstance(spec, np.ndarray) or isinstance(spec, (list, tuple)):
        arr = np.asarray(spec, dtype=np.int64)
        if arr.ndim == 1:
            arr = np.broadcast_to(arr, (batch, T))
        return np.ascontiguousarray(arr)
    par = np.empty((batch, T), dtype=np.int64)
    if spec == "chain":
        par[:, 0] = -1
        par[:, 1:] = np.arange(T - 1)
        return par
    if spec == "random":
        for b in range(batch):
            par[b, 0] = -1
            for i in range(1, T):
                par[b, i] = rng.integers(0, i)
        return par
    if spec == "star":
        par[:, 0] = -1
        par[:, 1:] = 0
        return par
    raise ValueError(f"unknown tree spec {spec!r}")


def make_inputs(*, batch, num_heads, prefix, T, tree="random", pool_slots, nsplit=64,
                seed=0, placement="scattered", softmax_scale=None, q_mode="normal",
                name="custom", poison=True, rows_per_table=None):
    """Draw one verify workload.

    prefix: "fixed:L", "uniform:lo:hi", or an explicit list of B lengths.
    tree: "chain", "random", "star", or an explicit [B, T] (or [T]) parent array.
    placement: "scattered" (random distinct slots) or "contiguous" (slots 0..n-1).
    q_mode: "normal" (N(0,1)) or "zero".
    poison: unused pool slots hold bf16 NaN (default) instead of zeros.
    """
    rng = np.random.default_rng(seed)
    L = _draw_prefix(rng, prefix, batch)
    if (L < 0).any():
        raise ValueError("prefix lengths must be >= 0")
    par = _draw_tree(rng, tree, batch, T)
    n = int(L.sum() + batch * T)
    if n > pool_slots:
        raise ValueError(f"{n} keys do not fit a {pool_slots}-slot pool")
    perm = rng.permutation(pool_slots)[:n]
    if placement == "scattered":
        slots = perm.astype(np.int64)
    elif placement == "contiguous":
        slots = np.arange(n, dtype=np.int64)
    else:
        raise ValueError(f"unknown placement {placement!r}")

    if q_mode == "normal":
        q = f32_to_bf16_bits(rng.standard_normal((batch * T, num_heads, D_QK), dtype=np.float32))
    elif q_mode == "zero":
        q = np.zeros((batch * T, num_heads, D_QK), dtype=np.uint16)
    else:
        raise ValueError(f"unknown q_mode {q_mode!r}")

    kv_pool = np.full((pool_slots, D_QK), BF16_NAN if poison else np.uint16(0), dtype=np.uint16)
    # Latent rows for the used keys, in logical order, written at their slots.
    step = 1 << 16
    for s in range(0, n, step):
        e = min(n, s + step)
        vals = rng.standard_normal((e - s, D_QK), dtype=np.float32)
        kv_pool[slots[s:e]] = f32_to_bf16_bits(vals)

    # Per-request slot lists: prefix slots in req_to_token, tree slots in
    # out_cache_loc (and also mirrored after the prefix in req_to_token, the
    # way an allocator records freshly written draft tokens).
    stride = int(L.max() + T) if batch > 0 else T
    R = rows_per_table if rows_per_table is not None else batch
    req_to_token = np.full((R, stride), -1, dtype=np.int32)
    # Request b lives in table row (B-1-b): a fixed, non-identity indirection.
    req_pool_indices = np.array([(R - 1 - b) for b in range(batch)], dtype=np.int32)
    out_cache_loc = np.empty(batch * T, dtype=np.int32)
    off = 0
    for b in range(batch):
        lb = int(L[b])
        row = req_pool_indices[b]
        req_to_token[row, :lb] = slots[off:off + lb]
        out_cache_loc[b * T:(b + 1) * T] = slots[off + lb:off + lb + T]
        req_to_token[row, lb:lb + T] = slots[off + lb:off + lb + T]
        off += lb + T

    scale = softmax_scale if softmax_scale is not None else 1.0 / np.sqrt(192.0)
    return VerifyInputs(
        name=name, batch=batch, num_heads=num_heads, T=T,
        prefix_lens=L.astype(np.int32), tree_parent=par.astype(np.int32),
        req_to_token=req_to_token, req_pool_indices=req_pool_indices,
        out_cache_loc=out_cache_loc, q=q, kv_pool=kv_pool, nsplit=nsplit,
        softmax_scale=float(scale), seed=seed, placement=placement,
    )


def make_config(idx: int, placement: str = "scattered", seed: int | None = None, **over):
    """One of the five named verify workloads (see CONFIGS)."""
    c = dict(CONFIGS[idx])
    c.update(over)
    return make_inputs(batch=c["batch"], num_heads=c["num_heads"], prefix=c["prefix"], T=c["T"],
                       tree=c["tree"], pool_slots=c["pool_slots"], nsplit=c["nsplit"],
                       seed=c["seed"] if seed is None else seed, placement=placement,
                       name=c["name"])


def make_sparse_decode(seed: int | None = None, **over):
    """The sparse-MLA decode workload (see SPARSE_DECODE)."""
    c = dict(SPARSE_DECODE)
    c.update(over)
    return make_inputs(batch=c["batch"], num_heads=c["num_heads"], prefix=c["prefix"], T=c["T"],
                       tree=c["tree"], pool_slots=c["pool_slots"], nsplit=c["nsplit"],
                       seed=c["seed"] if seed is None else seed, name=c["name"])


# ---------------------------------------------------------------- tree acceptance
@dataclass
class AcceptInputs:
    tree_parent: np.ndarray      # int32 [B, T], parent[0] = -1
    draft_tokens: np.ndarray     # int32 [B, T], token proposed at each node (node 0: last committed)
    target_argmax: np.ndarray    # int32 [B, T], the target model's greedy next token after each node
    out_cache_loc: np.ndarray    # int32 [B, T], KV slot of each node


def make_accept_inputs(*, batch, T, tree="random", vocab=32000, match=0.7, pool_slots=1 << 20,
                       seed=0):
    """Draft trees with tokens and target choices. At each node, with
    probability `match` the target's choice is the draft token of one of the
    node's children (drawn uniformly), else a random token."""
    rng = np.random.default_rng(seed)
    par = _draw_tree(rng, tree, batch, T).astype(np.int32)
    draft = rng.integers(0, vocab, size=(batch, T)).astype(np.int32)
    target = rng.integers(0, vocab, size=(batch, T)).astype(np.int32)
    for b in range(batch):
        for t in range(T):
            kids = np.nonzero(par[b] == t)[0]
            if kids.size and rng.random() < match:
                target[b, t] = draft[b, kids[rng.integers(0, kids.size)]]
    loc = rng.permutation(pool_slots)[:batch * T].reshape(batch, T).astype(np.int32)
    return AcceptInputs(par, draft, target, loc)


# ---------------------------------------------------------------- KV relocation
@dataclass
class RelocateInputs:
    kv_pool: np.ndarray          # uint16 (bf16 bits) [S, 576]
    req_to_token: np.ndarray     # int32 [R, stride]
    req_pool_indices: np.ndarray  # int32 [B]
    prefix_lens: np.ndarray      # int32 [B]
    dst_start: np.ndarray        # int32 [B], contiguous free destination range per request
    progress: np.ndarray         # int32 [B], rows already moved (0)


def make_relocate_inputs(*, batch, prefix, pool_slots, seed=0, poison=True, in_place=0):
    """Scattered live rows in the low part of the pool and, for every request,
    a contiguous free destination range in the top part. `in_place` rows at
    the start of request 0 already sit at their destination."""
    rng = np.random.default_rng(seed)
    L = _draw_prefix(rng, prefix, batch)
    total = int(L.sum())
    if 2 * total > pool_slots:
        raise ValueError("pool too small")
    top = pool_slots - total
    src = rng.permutation(top)[:total].astype(np.int64)
    dst_start = (top + np.concatenate([[0], np.cumsum(L)[:-1]])).astype(np.int32)
    if in_place and batch:
        k = min(in_place, int(L[0]))
        src[:k] = dst_start[0] + np.arange(k)
    kv_pool = np.full((pool_slots, D_QK), BF16_NAN if poison else np.uint16(0), dtype=np.uint16)
    kv_pool[src] = f32_to_bf16_bits(rng.standard_normal((total, D_QK), dtype=np.float32))
    stride = int(L.max()) if batch else 1
    req_to_token = np.full((batch, max(stride, 1)), -1, dtype=np.int32)
    rpi = np.array([batch - 1 - b for b in range(batch)], dtype=np.int32)
    off = 0
    for b in range(batch):
        req_to_token[rpi[b], :L[b]] = src[off:off + L[b]]
        off += int(L[b])
    return RelocateInputs(kv_pool, req_to_token, rpi, L.astype(np.int32), dst_start,
                          np.zeros(batch, dtype=np.int32))


# ---------------------------------------------------------------- fp8 paged MQA indexer
@dataclass
class IndexerInputs:
    q: np.ndarray            # uint8 fp8-e4m3 codes [B, H, 128]
    weights: np.ndarray      # float32 [B, H]
    kv_blocks: np.ndarray    # uint8 [nblocks, 8448]: 64 x 128 fp8 codes, then 64 fp32 scales
    block_table: np.ndarray  # int32 [B, max_pages]; -1 past a request's pages
    seq_lens: np.ndarray     # int32 [B]


def _e4m3_codes(rng, shape, emin=4, emax=9):
    """Random fp8-e4m3 codes with exponent field in [emin, emax] (magnitudes
    2^-3 .. ~2^3), random sign and mantissa; never the NaN codes."""
    s = rng.integers(0, 2, size=shape)
    e = rng.integers(emin, emax + 1, size=shape)
    m = rng.integers(0, 8, size=shape)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def make_indexer_inputs(*, batch, num_heads=64, seq_lens, max_pages, nblocks=None, seed=0):
    """Queries, per-head weights, paged fp8 keys with per-position fp32 scales
    and a page table of distinct physical blocks per request."""
    rng = np.random.default_rng(seed)
    lens = _draw_prefix(rng, seq_lens, batch).astype(np.int32)
    pages = (lens + 63) // 64
    if (pages > max_pages).any():
        raise ValueError("seq_lens exceed max_pages")
    need = int(pages.sum())
    nblocks = nblocks if nblocks is not None else max(need, 1)
    q = _e4m3_codes(rng, (batch, num_heads, 128))
    w = (rng.standard_normal((batch, num_heads)) / 8.0).astype(np.float32)
    kv = np.zeros((nblocks, 8448), dtype=np.uint8)
    kv[:, :8192] = _e4m3_codes(rng, (nblocks, 8192))
    scales = rng.uniform(0.5, 2.0, size=(nblocks, 64)).astype(np.float32) / 16.0
    kv[:, 8192:] = scales.view(np.uint8).reshape(nblocks, 256)
    perm = rng.permutation(nblocks)
    bt = np.full((batch, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(batch):
        bt[b, :pages[b]] = perm[off:off + pages[b]]
        off += int(pages[b])
    return IndexerInputs(q, w, kv, bt, lens)
