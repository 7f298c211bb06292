"""Seeded synthetic inputs shared by the CUDA path, the oracle and the benchmark.

This module only draws random numbers and arranges them in the shapes the
workloads need.  It performs none of the drafter or tree arithmetic: every
value it returns is an input (weights, target features, a cache prefix,
anchor tokens, logits, target tokens).  Both sides of a parity test receive
the same bytes from here.

Recipe (stands in for the pages' trained checkpoints and benchmark prompts,
which are not available):

* weights: i.i.d. N(0, 1/fan_in), embedding N(0, 1), norm gains 1, rounded to
  the workload dtype;
* target features: N(0, 1) of shape [rows, n_feat * d_feat];
* cache prefix for parity tests: N(0, 1) keys and values (a random injected
  context is itself Gaussian, so this matches the distribution of injected
  entries);
* anchors: uniform over the vocabulary without the mask token;
* stress logits: N(0, 2) (variance 2) in bf16, plus +8 on one planted token per
  (request, position);
* target tokens: drawn per tree node from a counter-based generator keyed by
  (seed, request, node), following the agreement rule of each workload.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np
import torch

from .configs import DrafterShape, Workload

_M64 = (1 << 64) - 1


def _torch_dtype(name: str) -> torch.dtype:
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919 + 12345) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal(shape: Sequence[int], std: float, seed: int, stream: int, device="cpu",
           dtype: str = "fp32") -> torch.Tensor:
    """N(0, std^2) samples, drawn in fp32 and rounded to `dtype`."""
    g = _gen(seed, stream, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(_torch_dtype(dtype))


def drafter_weights(shape: DrafterShape, seed: int, device="cpu") -> Dict[str, object]:
    """Random-init drafter weights in their natural [out, in] layout.

    Keys: w_proj [d, n_feat*d_feat], embed [V, d], lm_head [V, d], final_norm [d],
    and per layer (lists of length n_layers): attn_norm [d], wq [n_q*hd, d],
    wk [n_kv*hd, d], wv [n_kv*hd, d], wo [d, n_q*hd], uk [n_kv*hd, d],
    uv [n_kv*hd, d], mlp_norm [d], w_gate [d_ff, d], w_up [d_ff, d],
    w_down [d, d_ff].
    """
    s, dt = shape, shape.dtype
    fin = s.n_feat * s.d_feat
    qd, kd = s.n_q * s.head_dim, s.kv_dim
    stream = [0]

    def nrm(rows, cols, std):
        stream[0] += 1
        return normal((rows, cols), std, seed, stream[0], device, dt)

    def ones(n):
        return torch.ones(n, dtype=_torch_dtype(dt), device=device)

    w: Dict[str, object] = {
        "w_proj": nrm(s.d, fin, 1.0 / math.sqrt(fin)),
        "embed": nrm(s.vocab, s.d, 1.0),
        "lm_head": nrm(s.vocab, s.d, 1.0 / math.sqrt(s.d)),
        "final_norm": ones(s.d),
    }
    per = {k: [] for k in ("attn_norm", "wq", "wk", "wv", "wo", "uk", "uv",
                           "mlp_norm", "w_gate", "w_up", "w_down")}
    for _ in range(s.n_layers):
        per["attn_norm"].append(ones(s.d))
        per["wq"].append(nrm(qd, s.d, 1.0 / math.sqrt(s.d)))
        per["wk"].append(nrm(kd, s.d, 1.0 / math.sqrt(s.d)))
        per["wv"].append(nrm(kd, s.d, 1.0 / math.sqrt(s.d)))
        per["wo"].append(nrm(s.d, qd, 1.0 / math.sqrt(qd)))
        per["uk"].append(nrm(kd, s.d, 1.0 / math.sqrt(s.d)))
        per["uv"].append(nrm(kd, s.d, 1.0 / math.sqrt(s.d)))
        per["mlp_norm"].append(ones(s.d))
        per["w_gate"].append(nrm(s.d_ff, s.d, 1.0 / math.sqrt(s.d)))
        per["w_up"].append(nrm(s.d_ff, s.d, 1.0 / math.sqrt(s.d)))
        per["w_down"].append(nrm(s.d, s.d_ff, 1.0 / math.sqrt(s.d_ff)))
    w.update(per)
    return w


def random_gains(shape: DrafterShape, seed: int, device="cpu") -> Dict[str, object]:
    """Non-unit norm gains (U[0.5, 1.5]) for tests that must see the gain applied."""
    g = _gen(seed, 999, device)
    dt = _torch_dtype(shape.dtype)

    def one():
        return (0.5 + torch.rand(shape.d, generator=g, device=device)).to(dt)

    return {
        "final_norm": one(),
        "attn_norm": [one() for _ in range(shape.n_layers)],
        "mlp_norm": [one() for _ in range(shape.n_layers)],
    }


def tied_lm_head(shape: DrafterShape, seed: int, device="cpu") -> torch.Tensor:
    """An LM head [V, d] whose logits tie exactly, for tie-breaking tests.

    Row v has one nonzero entry, at a random column c(v), of value
    +-{1/4, 1/2, 1}: every logit is then a single product of the normed
    activation and a power of two (exact in fp32 whatever the summation
    order), so tokens that share (c, value) tie bit for bit, and they sit at
    random ids spread over the whole vocabulary."""
    g = _gen(seed, 998, device)
    cols = torch.randint(0, shape.d, (shape.vocab,), generator=g, device=device)
    mag = torch.randint(0, 3, (shape.vocab,), generator=g, device=device)
    sign = torch.randint(0, 2, (shape.vocab,), generator=g, device=device) * 2 - 1
    vals = sign.float() * torch.pow(2.0, -mag.float())
    w = torch.zeros(shape.vocab, shape.d, dtype=torch.float32, device=device)
    w[torch.arange(shape.vocab, device=device), cols] = vals
    return w.to(_torch_dtype(shape.dtype))


def features(n_rows: int, shape: DrafterShape, seed: int, stream: int = 100,
             device="cpu") -> torch.Tensor:
    """Target hidden features [n_rows, n_feat*d_feat], N(0, 1)."""
    return normal((n_rows, shape.n_feat * shape.d_feat), 1.0, seed, stream, device,
                  shape.dtype)


def cache_prefix(shape: DrafterShape, n_req: int, cap: int, seed: int,
                 device="cpu"):
    """Random injected-context entries: per layer K and V of [n_req, n_kv, cap, hd]."""
    ks, vs = [], []
    for layer in range(shape.n_layers):
        ks.append(normal((n_req, shape.n_kv, cap, shape.head_dim), 1.0, seed,
                         200 + 2 * layer, device, shape.dtype))
        vs.append(normal((n_req, shape.n_kv, cap, shape.head_dim), 1.0, seed,
                         201 + 2 * layer, device, shape.dtype))
    return ks, vs


def context_lengths(wl: Workload) -> np.ndarray:
    """Per-request context length: fixed, or U{lo..hi} (ragged serving batch)."""
    lo, hi = wl.ctx
    if lo == hi:
        return np.full(wl.n_req, lo, dtype=np.int32)
    rng = np.random.default_rng(wl.seed)
    return rng.integers(lo, hi + 1, size=wl.n_req).astype(np.int32)


def anchors(n_req: int, vocab: int, mask_id: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed + 77)
    a = rng.integers(0, vocab - 1, size=n_req)
    a = np.where(a >= mask_id, a + 1, a)   # skip the mask token
    return a.astype(np.int32)


def stress_logits(n_req: int, D: int, vocab: int, seed: int, device="cpu"):
    """bf16 logits [n_req*D, vocab] ~ N(0, 2) plus +8 on one planted token per row.

    Returns (logits, planted_ids[n_req*D]).
    """
    rows = n_req * D
    x = normal((rows, vocab), math.sqrt(2.0), seed, 300, device, "fp32")
    g = _gen(seed, 301, device)
    planted = torch.randint(0, vocab, (rows,), generator=g, device=device)
    idx = torch.arange(rows, device=device)
    x[idx, planted] += 8.0
    return x.to(torch.bfloat16), planted.to(torch.int32)


def random_topk_table(n_req: int, D: int, K: int, vocab: int, seed: int,
                      tie_fraction: float = 0.25):
    """A synthetic per-depth top-K table for tree tests.

    logp [n_req, D, K] fp32, non-positive and sorted descending; ids
    [n_req, D, K] int32, distinct within a row.  Consecutive values are spaced
    by exponential gaps; for a fraction of rows the gaps are rounded to a coarse
    grid (zero included) so that exact ties, the case bf16 logits produce, are
    exercised.
    """
    rng = np.random.default_rng(seed + 991)
    first = -rng.exponential(0.7, size=(n_req, D, 1)) - 0.05
    gaps = rng.exponential(0.8, size=(n_req, D, K - 1))
    coarse = rng.random((n_req, D, 1)) < tie_fraction
    gaps = np.where(coarse, np.round(gaps * 2.0) / 2.0, gaps)
    lp = np.concatenate([first, first - np.cumsum(gaps, axis=2)], axis=2)
    lp = np.ascontiguousarray(lp.astype(np.float32))
    ids = np.empty((n_req, D, K), dtype=np.int32)
    for r in range(n_req):
        for d in range(D):
            ids[r, d] = rng.choice(vocab, size=K, replace=False)
    return lp, ids


# ---------------------------------------------------------------------------
# Counter-based generator for target tokens (host only)
# ---------------------------------------------------------------------------

def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _M64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def counter_uniform(seed: int, req: int, node: int, k: int) -> float:
    """U[0,1) from splitmix64 applied to a key built from (seed, req, node, k)."""
    key = _splitmix64(seed & _M64)
    key = _splitmix64(key ^ ((req * 0x100000001B3) & _M64))
    key = _splitmix64(key ^ ((node * 0xD6E8FEB86659FD93) & _M64))
    key = _splitmix64(key ^ k)
    return (key >> 11) * (1.0 / (1 << 53))


def target_tokens(n_nodes: Sequence[int], depth: np.ndarray, topk_logp: np.ndarray,
                  topk_ids: np.ndarray, vocab: int, agree: float, seed: int,
                  temperature: float = 0.0,
                  preferred: Optional[np.ndarray] = None) -> np.ndarray:
    """Synthetic target-model token at every tree node (the target is not available).

    For a node of depth d < D the target's next token is drawn as follows.
    Greedy (temperature 0): with probability agree**(d+1) it is the preferred
    token at draft position d+1 (the drafter's top-1 unless `preferred`
    [n_req, D] names another, e.g. the planted token); otherwise it is drawn
    from q_{d+1} restricted to the other tokens, where q is known only on the
    top-K and the remaining mass stands for "some token outside the top-K"
    (drawn uniformly among the ids not in the table).  Temperature 1: drawn
    from q_{d+1} itself.  Nodes at depth D get a uniform token.
    Returns int32 [n_req, B+1] (entries past a tree's last node are -1).
    """
    n_req, D, K = topk_logp.shape
    width = depth.shape[1]
    out = np.full((n_req, width), -1, dtype=np.int32)
    for r in range(n_req):
        for n in range(int(n_nodes[r]) + 1):
            d = int(depth[r, n])
            if d >= D:
                u = counter_uniform(seed, r, n, 0)
                out[r, n] = min(int(u * vocab), vocab - 1)
                continue
            ids = [int(v) for v in topk_ids[r, d]]
            q = np.exp(topk_logp[r, d].astype(np.float64))
            pref = ids[0] if preferred is None else int(preferred[r, d])
            u0 = counter_uniform(seed, r, n, 0)
            if temperature == 0.0:
                if u0 < agree ** (d + 1):
                    out[r, n] = pref
                    continue
                w = np.array([0.0 if ids[k] == pref else q[k] for k in range(K)])
            else:
                w = q.copy()
            rest = max(0.0, 1.0 - float(q.sum()))   # mass outside the top-K
            total = float(w.sum()) + rest
            u1 = counter_uniform(seed, r, n, 1) * total
            acc = 0.0
            pick = None
            for k in range(K):
                acc += w[k]
                if u1 < acc:
                    pick = ids[k]
                    break
            if pick is None:
                excluded = set(ids) | {pref}
                j = 2
                while True:
                    cand = min(int(counter_uniform(seed, r, n, j) * vocab), vocab - 1)
                    if cand not in excluded:
                        pick = cand
                        break
                    j += 1
            out[r, n] = pick
    return out


# ---------------------------------------------------------------------------
# Device-side stand-in for the target's choices (graph-capturable)
# ---------------------------------------------------------------------------

def target_first_child(n_nodes: torch.Tensor, tok: torch.Tensor, parent: torch.Tensor,
                       vocab: int, agree_pct: int = 90) -> torch.Tensor:
    """target_tok [n_req, B+1] for a flattened tree: at node i the token of its
    first child in pop order (its best-scored child) when a multiplicative hash
    of that child's token falls below agree_pct percent, else that token + 1
    (or, at a leaf, the node's token + 1) modulo vocab, so walks stop at
    data-dependent depths (each step agrees with probability about agree_pct
    percent over random tokens) and the bonus token is always a valid id.
    Torch ops only, so a cycle that calls it can be captured in a CUDA graph."""
    n_req, W = tok.shape
    idx = torch.arange(W, device=tok.device).expand(n_req, W)
    valid = (idx >= 1) & (idx <= n_nodes.long()[:, None])
    par = torch.where(valid, parent.long(), torch.full_like(idx, W))
    first = torch.full((n_req, W + 1), W, dtype=torch.long, device=tok.device)
    first.scatter_reduce_(1, par, torch.where(valid, idx, torch.full_like(idx, W)), reduce="amin")
    first = first[:, :W]
    child_tok = torch.gather(tok.long(), 1, first.clamp(max=W - 1))
    has_child = first < W
    h = (child_tok * 2654435761).remainder(1 << 32) // 65536
    agree = has_child & (h.remainder(100) < agree_pct)
    other = (torch.where(has_child, child_tok, tok.long()) + 1).remainder(vocab)
    return torch.where(agree, child_tok, other).to(torch.int32)
