"""DDTree tree construction, tree mask and verifier walk (oracle; test infra only).

Source: "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
(the DDTree page).

* 3.4.3: a draft tree is a prefix-closed set of at most B non-root nodes; the
  surrogate objective is E_Q[alpha_T] = sum over nodes u of q(u) (Prop. 1) and
  the optimum is the top-B prefixes under the factorised Q (Prop. 2).
* 3.4.4, Algorithm 1: rank tuples rho over the per-depth top-K lists, score
  sigma(rho) = sum of the log-probabilities of its ranks, a max-heap seeded
  with (1); each pop becomes a tree node and pushes its next sibling (last rank
  + 1, if <= K) and its first child (append rank 1, if depth < depth limit);
  stop after B pops or when the heap is empty.
* 3.4.5: position id = depth; ancestor-only attention mask; the verifier walk
  follows the child whose token equals the target's choice at the current
  node, and the target's choice where it stops is the next bonus token.

Readings (the pages leave these open):
* a candidate's score is score(parent node) + logp[depth][rank], one float32
  addition of float32 values.  This equals the page's incremental sibling
  update mathematically and is reproducible bit for bit;
* ties in score pop in creation order (a counter over pushes; at each pop the
  sibling is created before the child);
* ranks and depths are 1-based as on the page; the root (the bonus token) is
  node 0 with depth 0 and rank 0; nodes 1..n are numbered in pop order;
* mask row i has bit j set iff node j is node i or an ancestor of i (the root
  included); rows and node entries past the last node are 0 / -1.
"""
from __future__ import annotations

import heapq
from typing import Dict

import numpy as np


def _f32(x) -> np.float32:
    return np.float32(x)


def build_tree(topk_logp, topk_ids, root_tok: int, B: int,
               depth_limit: int = None) -> Dict[str, object]:
    """Algorithm 1 for one request.

    topk_logp: [D, K] log q_i of the rank-k token at depth i (descending per row);
    topk_ids:  [D, K] the matching token ids.
    Returns dict with n_nodes, tok, parent, depth, rank, score (float32),
    mask (uint32 [B+1, ceil((B+1)/32)]) and instrumentation (pops, pushes,
    max_heap, pop_scores).
    """
    lp = np.asarray(topk_logp, dtype=np.float32)
    ids = np.asarray(topk_ids)
    D, K = lp.shape
    if depth_limit is not None:
        D = min(D, depth_limit)
    width = B + 1
    tok = np.full(width, -1, dtype=np.int32)
    parent = np.full(width, -1, dtype=np.int32)
    depth = np.full(width, -1, dtype=np.int32)
    rank = np.full(width, -1, dtype=np.int32)
    score = np.full(width, np.nan, dtype=np.float32)
    tok[0], depth[0], rank[0], score[0] = root_tok, 0, 0, _f32(0.0)

    heap = []
    seq = 0
    pushes = 0
    pop_scores = []
    if B > 0 and D > 0 and K > 0:
        s = _f32(score[0] + lp[0, 0]) + _f32(0.0)
        heapq.heappush(heap, (-float(s), seq, 0, 1, 1))
        seq += 1
        pushes += 1
    max_heap = len(heap)
    n = 0
    while n < B and heap:
        neg, _, p, d, r = heapq.heappop(heap)
        n += 1
        tok[n] = ids[d - 1, r - 1]
        parent[n], depth[n], rank[n] = p, d, r
        score[n] = _f32(-neg)
        pop_scores.append(score[n])
        if r < K:                                   # next sibling
            s = _f32(score[p] + lp[d - 1, r]) + _f32(0.0)
            heapq.heappush(heap, (-float(s), seq, p, d, r + 1))
            seq += 1
            pushes += 1
        if d < D:                                   # first child
            s = _f32(score[n] + lp[d, 0]) + _f32(0.0)
            heapq.heappush(heap, (-float(s), seq, n, d + 1, 1))
            seq += 1
            pushes += 1
        max_heap = max(max_heap, len(heap))

    return {
        "n_nodes": n, "tok": tok, "parent": parent, "depth": depth, "rank": rank,
        "score": score, "mask": tree_mask(parent, n, B),
        "pops": n, "pushes": pushes, "max_heap": max_heap,
        "pop_scores": np.array(pop_scores, dtype=np.float32),
    }


def tree_mask(parent, n_nodes: int, B: int) -> np.ndarray:
    """Ancestor-only attention mask, bit-packed: [B+1, ceil((B+1)/32)] uint32."""
    width = B + 1
    words = (width + 31) // 32
    mask = np.zeros((width, words), dtype=np.uint32)
    for i in range(n_nodes + 1):
        j = i
        while j >= 0:
            mask[i, j // 32] |= np.uint32(1 << (j % 32))
            j = int(parent[j]) if j > 0 else -1
    return mask


def rank_tuple(parent, rank, node: int):
    """The rank tuple (rho_1, ..., rho_d) of a node, read along its ancestors."""
    out = []
    j = node
    while j > 0:
        out.append(int(rank[j]))
        j = int(parent[j])
    return tuple(reversed(out))


def prefix_tokens(topk_ids, rho):
    """Token prefix (v_1^(rho_1), ..., v_d^(rho_d)) named by a rank tuple."""
    return tuple(int(topk_ids[i][r - 1]) for i, r in enumerate(rho))


def expected_acceptance(tree: Dict[str, object], topk_logp) -> float:
    """Prop. 1: E_Q[alpha_T] = sum over non-root nodes of q(u), in float64."""
    lp = np.asarray(topk_logp, dtype=np.float64)
    total = 0.0
    for i in range(1, tree["n_nodes"] + 1):
        rho = rank_tuple(tree["parent"], tree["rank"], i)
        total += float(np.exp(sum(lp[d, r - 1] for d, r in enumerate(rho))))
    return total


def accept_walk(tok, parent, n_nodes: int, target_tok, depth_cap: int):
    """Greedy verifier walk (DDTree page 3.4.5).

    Start at the root; while the current node has a child whose token equals
    target_tok[current], move to it.  Returns (accept_len, accepted_nodes padded
    with -1 to depth_cap, bonus = target_tok at the stop node).
    """
    node = 0
    path = []
    while True:
        y = int(target_tok[node])
        nxt = -1
        for c in range(1, n_nodes + 1):
            if int(parent[c]) == node and int(tok[c]) == y:
                nxt = c
                break
        if nxt < 0:
            break
        path.append(nxt)
        node = nxt
    accepted = np.full(depth_cap, -1, dtype=np.int32)
    accepted[:len(path)] = path
    return len(path), accepted, int(target_tok[node])
