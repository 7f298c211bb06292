"""Verification-side tree attention (oracle; test infrastructure only).

Source: "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
(the DDTree page), 3.4.5: the tree is flattened, every node's position id is
its depth, and under the ancestor-only mask a node attends to the past context
(the KV cache), to the root, to its ancestors and to itself, and to no other
tree node.  One attention layer of the target model over that sequence.

Readings (the page leaves these open): position ids are absolute, ctx_len +
depth (the root, at depth 0, takes the first position after the context);
grouped-query heads read KV head h // (n_q / n_kv); the rotary embedding is the
rotate-half form used for the drafter; rows of nodes past the last one are
zero.  Everything in float64.
"""
from __future__ import annotations

import math

import numpy as np

from oracle.drafter import apply_rope, f64


def tree_rope(x, ctx_len: int, depth, theta: float) -> np.ndarray:
    """x [B+1, heads, hd]: rows with depth >= 0 rotated at ctx_len + depth."""
    x = f64(x).copy()
    depth = np.asarray(depth)
    live = depth >= 0
    if live.any():
        x[live] = apply_rope(x[live], ctx_len + depth[live], theta)
    return x


def ancestors(mask_row, width: int):
    """Node indices whose bit is set in one bit-packed mask row."""
    return [j for j in range(width) if (int(mask_row[j // 32]) >> (j % 32)) & 1]


def tree_attention(q, k_tree, v_tree, cache_k, cache_v, ctx_len: int, mask, n_nodes: int,
                   n_q: int, n_kv: int) -> np.ndarray:
    """One request.

    q [B+1, n_q, hd] (rotated), k_tree / v_tree [B+1, n_kv, hd] (k rotated),
    cache_k / cache_v [n_kv, cap, hd], mask [B+1, W] uint32.
    out[i, h] = sum_j softmax_j(q[i, h] . key_j / sqrt(hd)) value_j over the
    context slots t < ctx_len and the tree nodes j in mask row i.
    """
    q, k_tree, v_tree = f64(q), f64(k_tree), f64(v_tree)
    ck, cv = f64(cache_k), f64(cache_v)
    width, _, hd = q.shape
    G = n_q // n_kv
    out = np.zeros_like(q)
    for i in range(n_nodes + 1):
        anc = ancestors(mask[i], width)
        for h in range(n_q):
            g = h // G
            keys = np.concatenate([ck[g, :ctx_len], k_tree[anc, g]], axis=0)
            vals = np.concatenate([cv[g, :ctx_len], v_tree[anc, g]], axis=0)
            s = keys @ q[i, h] / math.sqrt(hd)
            s = s - s.max()
            p = np.exp(s)
            out[i, h] = (p / p.sum()) @ vals
    return out
