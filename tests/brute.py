"""Brute-force per-row reference for tiny inputs, in pure Python.

Independent of the C oracle: it starts from the raw inputs (req_to_token,
out_cache_loc, tree_parent), walks the tree itself, and uses math.fsum for
every sum. Used only to pin the oracle on inputs small enough for Python
loops.
"""

import math

from workloads import bf16_bits_to_f32


def visible_slots(inp, b, t):
    """Pool slots a tree token (b, t) may attend to, in logical key order."""
    T = inp.T
    L = int(inp.prefix_lens[b])
    row = inp.req_to_token[int(inp.req_pool_indices[b])]
    slots = [int(row[j]) for j in range(L)]
    on_path = set()
    v = t
    while v != -1:
        on_path.add(v)
        v = int(inp.tree_parent[b, v])
    slots += [int(inp.out_cache_loc[b * T + u]) for u in range(T) if u in on_path]
    return slots


def brute_row(inp, n):
    H, T = inp.num_heads, inp.T
    h = n % H
    bt = n // H
    b, t = bt // T, bt % T
    q = [float(x) for x in bf16_bits_to_f32(inp.q[bt, h])]
    rows = [[float(x) for x in bf16_bits_to_f32(inp.kv_pool[s])] for s in visible_slots(inp, b, t)]
    scores = [inp.softmax_scale * math.fsum(q[d] * k[d] for d in range(576)) for k in rows]
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    Z = math.fsum(w)
    out = [math.fsum(w[i] * rows[i][d] for i in range(len(rows))) / Z for d in range(512)]
    return out, m + math.log(Z)
