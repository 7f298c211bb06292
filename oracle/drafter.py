"""The DFlash drafter pass, restated plainly (oracle; test infrastructure only).

Sources, cited by page title and section:

* "DFlash: Block Diffusion for Flash Speculative Decoding" (the DFlash page):
  3.4.3 feature fusion h_fused = W_proj [h_l1; ...; h_l5] and KV injection
  K = U_K h_fused, V = U_V h_fused stored as extra key/value pairs of every
  drafter layer; 3.4.4 the block [anchor, mask x (gamma-1)], bidirectional
  attention inside the block plus attention to the injected context, one
  forward pass, logits from the shared LM head.
* "Accelerating Speculative Decoding with Block Diffusion Draft Trees" (the
  DDTree page): 3.4.2 per-position marginals q_i = softmax(l_i).

Readings where the pages are silent (each is listed in the design notes):
pre-norm RMSNorm with a gain vector before attention, before the MLP and
before the LM head; rotate-half rotary embedding at absolute positions
(context slot t has position t, block row j has position ctx_len + j); no
biases, no QK-norm; SwiGLU MLP; grouped-query attention with query head h
reading key/value head h // (n_q / n_kv); by default every block row attends
to the whole context and the whole block (the anchor-isolated variant of the
DFlash page's 3.4.4 bullet list is available with ``anchor_sees_block=False``).

Everything is computed in float64 on whatever values are passed in (the tests
pass the exact bf16 or fp32 weight values upcast to float64).
"""
from __future__ import annotations

import math
from typing import Dict, Sequence

import numpy as np


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# Elementary layers (textbook definitions)
# ---------------------------------------------------------------------------

def rms_norm(x, gain, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis."""
    x = f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * f64(gain)


def rope_angles(pos, head_dim: int, theta: float) -> np.ndarray:
    """angle[p, i] = pos[p] * theta^(-2i/head_dim), i < head_dim/2."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return np.outer(f64(pos), inv_freq)


def apply_rope(x, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding.  x: [n, heads, hd], pos: [n].

    Dimension i (i < hd/2) pairs with i + hd/2 and the pair is rotated by
    angle[p, i]: (a, b) -> (a cos - b sin, b cos + a sin).
    """
    x = f64(x)
    hd = x.shape[-1]
    half = hd // 2
    ang = rope_angles(pos, hd, theta)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(x) -> np.ndarray:
    x = f64(x)
    return x / (1.0 + np.exp(-x))


def attention(q, k, v) -> np.ndarray:
    """softmax(q k^T / sqrt(hd)) v, with the softmax over all keys.

    q: [m, hd], k: [s, hd], v: [s, hd]  ->  [m, hd].
    """
    q, k, v = f64(q), f64(k), f64(v)
    scores = q @ k.T / math.sqrt(q.shape[-1])
    scores = scores - scores.max(axis=1, keepdims=True)
    p = np.exp(scores)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ v


# ---------------------------------------------------------------------------
# Step a1/a2: feature fusion and KV injection (DFlash page, 3.4.3)
# ---------------------------------------------------------------------------

def fuse_features(feats, w_proj) -> np.ndarray:
    """h_fused(t) = W_proj [h_l1(t); ...; h_ln(t)] for each injected position t.

    feats: [n, n_feat*d_feat] (the target layers' hidden states, concatenated),
    w_proj: [d, n_feat*d_feat]  ->  [n, d].
    """
    return f64(feats) @ f64(w_proj).T


def inject_kv(f, uk, uv, pos, n_kv: int, head_dim: int, theta: float):
    """One layer's injected context entries for positions `pos`.

    K_t = RoPE(U_K f_t, t), V_t = U_V f_t; returns (K, V) of [n_kv, n, hd],
    i.e. already laid out as the cache slots for those positions.
    """
    f = f64(f)
    n = f.shape[0]
    k = (f @ f64(uk).T).reshape(n, n_kv, head_dim)
    k = apply_rope(k, pos, theta)
    v = (f @ f64(uv).T).reshape(n, n_kv, head_dim)
    return k.transpose(1, 0, 2), v.transpose(1, 0, 2)


# ---------------------------------------------------------------------------
# Steps a3-a5: the block pass (DFlash page, 3.4.4)
# ---------------------------------------------------------------------------

def _w(weights, name, layer=None):
    obj = weights[name] if layer is None else weights[name][layer]
    return f64(obj)


def drafter_block(weights: Dict, dims: Dict, cache_k: Sequence, cache_v: Sequence,
                  ctx_len: int, anchor: int, L: int,
                  anchor_sees_block: bool = True, vocab_chunk: int = 16384,
                  return_hidden: bool = False, return_residual: bool = False):
    """Logits of the L-1 mask positions for one request.

    dims: n_layers, d, n_q, n_kv, head_dim, vocab, mask_id, rope_theta, rms_eps.
    cache_k[l], cache_v[l]: [n_kv, >= ctx_len, hd] injected context of layer l.
    Returns logits [L-1, V] (float64); with return_hidden also the final
    normalised hidden rows [L-1, d]; with return_residual also the residual
    stream of all L rows before the final norm.
    """
    nl, d = dims["n_layers"], dims["d"]
    n_q, n_kv, hd = dims["n_q"], dims["n_kv"], dims["head_dim"]
    theta, eps = dims["rope_theta"], dims["rms_eps"]
    group = n_q // n_kv

    embed = weights["embed"]
    x = np.stack([f64(embed[int(anchor)])] +
                 [f64(embed[int(dims["mask_id"])])] * (L - 1))      # [L, d]
    pos = ctx_len + np.arange(L)

    for l in range(nl):
        h = rms_norm(x, _w(weights, "attn_norm", l), eps)
        q = (h @ _w(weights, "wq", l).T).reshape(L, n_q, hd)
        kb = (h @ _w(weights, "wk", l).T).reshape(L, n_kv, hd)
        vb = (h @ _w(weights, "wv", l).T).reshape(L, n_kv, hd)
        q = apply_rope(q, pos, theta)
        kb = apply_rope(kb, pos, theta)
        ck, cv = f64(cache_k[l]), f64(cache_v[l])
        o = np.empty((L, n_q, hd))
        for hq in range(n_q):
            g = hq // group
            keys = np.concatenate([ck[g, :ctx_len], kb[:, g]], axis=0)
            vals = np.concatenate([cv[g, :ctx_len], vb[:, g]], axis=0)
            if anchor_sees_block:
                o[:, hq] = attention(q[:, hq], keys, vals)
            else:
                # the anchor row sees the context and itself only
                o[0, hq] = attention(q[0:1, hq], keys[:ctx_len + 1],
                                     vals[:ctx_len + 1])[0]
                o[1:, hq] = attention(q[1:, hq], keys, vals)
        x = x + o.reshape(L, n_q * hd) @ _w(weights, "wo", l).T
        h = rms_norm(x, _w(weights, "mlp_norm", l), eps)
        gate = h @ _w(weights, "w_gate", l).T
        up = h @ _w(weights, "w_up", l).T
        x = x + (silu(gate) * up) @ _w(weights, "w_down", l).T

    hf = rms_norm(x[1:], _w(weights, "final_norm"), eps)            # [L-1, d]
    lm = weights["lm_head"]
    V = dims["vocab"]
    logits = np.empty((L - 1, V))
    for v0 in range(0, V, vocab_chunk):
        v1 = min(V, v0 + vocab_chunk)
        logits[:, v0:v1] = hf @ f64(lm[v0:v1]).T
    if return_hidden:
        return logits, hf
    if return_residual:
        return logits, x
    return logits


# ---------------------------------------------------------------------------
# Step a6: marginals, log-softmax and top-K (DDTree page, 3.4.2 and 3.4.4)
# ---------------------------------------------------------------------------

def log_softmax(logits):
    """log q_i(v) = l_iv - log sum_v exp(l_iv), per row.  Returns (logp, lse)."""
    x = f64(logits)
    m = x.max(axis=-1, keepdims=True)
    lse = m + np.log(np.exp(x - m).sum(axis=-1, keepdims=True))
    return x - lse, lse[..., 0]


def topk(values, K: int):
    """The K largest entries of each row, ordered by (value desc, index asc).

    values: [rows, V]  ->  (ids int32 [rows, K], vals float64 [rows, K]).
    Equal values are ordered by the lower token id first.
    """
    x = f64(values)
    rows, V = x.shape
    ids = np.empty((rows, K), dtype=np.int32)
    vals = np.empty((rows, K))
    for r in range(rows):
        row = x[r]
        kth = np.partition(row, V - K)[V - K]          # K-th largest value
        cand = np.nonzero(row >= kth)[0]
        order = np.lexsort((cand, -row[cand]))[:K]
        ids[r] = cand[order]
        vals[r] = row[cand[order]]
    return ids, vals


def logits_topk(logits, K: int):
    """Top-K token ids with their log-probabilities, per row.

    Returns (ids [rows, K], logp [rows, K], lse [rows]) with logp = logit - lse.
    """
    x = f64(logits)
    m = x.max(axis=-1, keepdims=True)
    lse = (m + np.log(np.exp(x - m).sum(axis=-1, keepdims=True)))[:, 0]
    ids, vals = topk(x, K)
    return ids, vals - lse[:, None], lse
