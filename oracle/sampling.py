"""Vanilla DFlash drafting at temperature T and its chain tree (oracle; test
infrastructure only).

Source: "DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.4
(the drafted token of a block position is the argmax of its logits at
temperature 0, a sample from softmax(logits) at temperature 1) and 3.4.1 (the
drafted block is verified as one chain: accept up to the first mismatch).

Readings (the page names no sampler):
* a sample from softmax(l / T) is drawn with the Gumbel-max rule: the token
  maximising l_v / T + G_v with G_v = -log(-log U_v) and U_v uniform on (0, 1);
* U_v comes from the counter-based SplitMix64 generator (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", 2014): the k-th output of
  the generator seeded with `seed` is mix(seed + k * 0x9E3779B97F4A7C15), with
  mix(z) = z ^ z >> 30, * 0xBF58476D1CE4E5B9, ^ >> 27, * 0x94D049BB133111EB,
  ^ >> 31 (all mod 2^64); element v of row r takes k = (r << 32 | v) + 1 and
  U = (top 23 bits + 0.5) / 2^23, exact in float32 and strictly inside (0, 1)
  (with 24 bits the largest value rounds to 1 in float32 and G becomes
  infinite);
* the decision is taken in float32: s_v = f32(l_v) * f32(1 / T) + G_v with G
  evaluated in float32, ties to the smaller token id; T = 0 is the argmax;
* the K best scores (score desc, id asc) are a draw of K tokens without
  replacement (the Gumbel-top-k property), and the log-probability reported
  for a drawn token is log softmax(l)[token];
* the chain tree of a drafted block: node 0 the anchor, node d the token of
  position d (rank 1: entry 0 of the position's list), each node the parent
  of the next, the ancestor mask of a chain (row i: bits 0..i); a budget
  B < D keeps the first B positions.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def splitmix64(seed: int, k: int) -> int:
    """k-th output (k >= 1) of SplitMix64 seeded with `seed` (Python integers)."""
    z = (seed + k * GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def splitmix64_np(seed: int, k: np.ndarray) -> np.ndarray:
    """The same over a uint64 array of counters (wrapping uint64 arithmetic)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + k.astype(np.uint64) * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def uniforms(seed: int, row: int, vocab: int) -> np.ndarray:
    """U_v for v < vocab of one row, float32 in (0, 1)."""
    k = (np.uint64(row) << np.uint64(32)) | np.arange(vocab, dtype=np.uint64)
    x = splitmix64_np(seed, k + np.uint64(1))
    top = (x >> np.uint64(41)).astype(np.float64)
    return ((top + 0.5) * 2.0 ** -23).astype(np.float32)


def gumbel(u: np.ndarray) -> np.ndarray:
    """G = -log(-log U), in float32."""
    u = np.asarray(u, dtype=np.float32)
    return -np.log(-np.log(u))


def scores(logits_row, temperature: float, seed: int, row: int) -> np.ndarray:
    """s_v = f32(l_v) * f32(1/T) + G_v (float32)."""
    l = np.asarray(logits_row, dtype=np.float32)
    inv_t = np.float32(1.0 / temperature)
    return l * inv_t + gumbel(uniforms(seed, row, l.shape[0]))


def sample_rows(logits, temperature: float, seed: int, row_offset: int = 0) -> np.ndarray:
    """Token per row: argmax of the row (T == 0) or of its Gumbel scores;
    ties to the smaller id (np.argmax takes the first maximum)."""
    logits = np.asarray(logits, dtype=np.float32)
    out = np.empty(logits.shape[0], dtype=np.int32)
    for r in range(logits.shape[0]):
        s = logits[r] if temperature == 0 else scores(logits[r], temperature, seed,
                                                     row_offset + r)
        out[r] = int(np.argmax(s))
    return out


def gumbel_topk(logits_row, temperature: float, seed: int, row: int, K: int):
    """The K best Gumbel scores of one row: ids (score desc, id asc) and the
    log-probabilities log softmax(l) of those ids (float64)."""
    l = np.asarray(logits_row, dtype=np.float32)
    s = scores(l, temperature, seed, row)
    order = np.lexsort((np.arange(s.shape[0]), -s.astype(np.float64)))[:K]
    l64 = l.astype(np.float64)
    m = l64.max()
    lse = m + np.log(np.sum(np.exp(l64 - m)))
    return order.astype(np.int32), l64[order] - lse


def chain_tree(root_tok: int, tokens, B: int):
    """Flattened chain tree of the drafted tokens in buffers of width B + 1:
    tok, parent, depth, rank, mask like the DDTree oracle's build_tree output,
    n_nodes = min(len(tokens), B)."""
    D = min(len(tokens), B)
    width = B + 1
    tok = np.full(width, -1, dtype=np.int32)
    parent = np.full(width, -1, dtype=np.int32)
    depth = np.full(width, -1, dtype=np.int32)
    rank = np.full(width, -1, dtype=np.int32)
    tok[0], depth[0], rank[0] = root_tok, 0, 0
    for d in range(1, D + 1):
        tok[d], parent[d], depth[d], rank[d] = tokens[d - 1], d - 1, d, 1
    words = (width + 31) // 32
    mask = np.zeros((width, words), dtype=np.uint32)
    for i in range(D + 1):
        for j in range(i + 1):
            mask[i, j // 32] |= np.uint32(1 << (j % 32))
    return dict(n_nodes=D, tok=tok, parent=parent, depth=depth, rank=rank, mask=mask)
