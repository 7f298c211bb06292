"""Pins for the tree-attention oracle (DDTree page, 3.4.5): a chain tree is
ordinary causal attention over [context; chain] (checked against a masked
matrix softmax written independently here), every branch of a star sees only
the root and itself, the root sees only the context and itself, rows past the
last node are zero, and depth position ids reduce to sequential positions on
a chain and to equal rotations at equal depths."""
import math

import numpy as np

from oracle import ddtree as odt
from oracle import drafter as od
from oracle import verify as ov


def _causal_reference(q_seq, k_seq, v_seq):
    """Masked matrix softmax over one head: row i sees keys 0..i (a lower-
    triangular mask), computed with a log-sum-exp normaliser."""
    s = q_seq @ k_seq.T / math.sqrt(q_seq.shape[-1])
    n, m = s.shape
    allowed = np.tril(np.ones((n, m), dtype=bool), k=m - n)
    s = np.where(allowed, s, -np.inf)
    lse = np.log(np.sum(np.exp(s - s.max(axis=1, keepdims=True)), axis=1, keepdims=True)) + \
        s.max(axis=1, keepdims=True)
    return np.exp(s - lse) @ v_seq


def _problem(seed, B, ctx, n_q=4, n_kv=2, hd=8, cap=None):
    rng = np.random.default_rng(seed)
    cap = cap or ctx + 3
    q = rng.normal(size=(B + 1, n_q, hd))
    kt = rng.normal(size=(B + 1, n_kv, hd))
    vt = rng.normal(size=(B + 1, n_kv, hd))
    ck = rng.normal(size=(n_kv, cap, hd))
    cv = rng.normal(size=(n_kv, cap, hd))
    return q, kt, vt, ck, cv


def test_chain_tree_is_causal_attention():
    B, ctx, n_q, n_kv = 9, 13, 4, 2
    q, kt, vt, ck, cv = _problem(1, B, ctx, n_q, n_kv)
    parent = np.array([-1] + list(range(B)))
    mask = odt.tree_mask(parent, B, B)
    out = ov.tree_attention(q, kt, vt, ck, cv, ctx, mask, B, n_q, n_kv)
    G = n_q // n_kv
    for h in range(n_q):
        g = h // G
        keys = np.concatenate([ck[g, :ctx], kt[:, g]])
        vals = np.concatenate([cv[g, :ctx], vt[:, g]])
        ref = _causal_reference(q[:, h], keys, vals)
        assert np.allclose(out[:, h], ref, atol=1e-12, rtol=0)


def test_star_branches_see_only_root_and_themselves():
    B, ctx, n_q, n_kv = 6, 5, 2, 1
    q, kt, vt, ck, cv = _problem(2, B, ctx, n_q, n_kv)
    parent = np.array([-1] + [0] * B)
    mask = odt.tree_mask(parent, B, B)
    out = ov.tree_attention(q, kt, vt, ck, cv, ctx, mask, B, n_q, n_kv)
    for i in range(1, B + 1):
        for h in range(n_q):
            keys = np.concatenate([ck[0, :ctx], kt[[0, i], 0]])
            vals = np.concatenate([cv[0, :ctx], vt[[0, i], 0]])
            ref = _causal_reference(q[[i], h], keys, vals)
            assert np.allclose(out[i, h], ref[0], atol=1e-12, rtol=0)
    # changing another branch's key or value leaves node 1 alone
    kt2, vt2 = kt.copy(), vt.copy()
    kt2[2] += 5.0
    vt2[3] -= 7.0
    out2 = ov.tree_attention(q, kt2, vt2, ck, cv, ctx, mask, B, n_q, n_kv)
    assert np.array_equal(out2[1], out[1])


def test_root_only_and_rows_past_the_last_node():
    B, ctx = 5, 4
    q, kt, vt, ck, cv = _problem(3, B, ctx, 2, 2)
    parent = np.array([-1, 0, 1, -1, -1, -1])
    mask = odt.tree_mask(parent, 2, B)
    out = ov.tree_attention(q, kt, vt, ck, cv, ctx, mask, 2, 2, 2)
    assert np.all(out[3:] == 0)
    for h in range(2):
        keys = np.concatenate([ck[h, :ctx], kt[[0], h]])
        vals = np.concatenate([cv[h, :ctx], vt[[0], h]])
        ref = _causal_reference(q[[0], h], keys, vals)
        assert np.allclose(out[0, h], ref[0], atol=1e-12, rtol=0)


def test_no_context_root_returns_its_own_value():
    q, kt, vt, ck, cv = _problem(4, 0, 0, 2, 1)
    mask = odt.tree_mask(np.array([-1]), 0, 0)
    out = ov.tree_attention(q, kt, vt, ck, cv, 0, mask, 0, 2, 1)
    for h in range(2):
        assert np.allclose(out[0, h], vt[0, 0], atol=1e-14)


def test_depth_positions():
    rng = np.random.default_rng(5)
    ctx, theta = 37, 1e6
    x = rng.normal(size=(7, 3, 8))
    chain_depth = np.arange(7)
    assert np.allclose(ov.tree_rope(x, ctx, chain_depth, theta),
                       od.apply_rope(x, ctx + np.arange(7), theta), atol=1e-14)
    # equal content at equal depth on two branches rotates identically; a row
    # past the last node (depth -1) is left as it is
    x[2] = x[1]
    depth = np.array([0, 1, 1, 2, 2, 3, -1])
    y = ov.tree_rope(x, ctx, depth, theta)
    assert np.array_equal(y[1], y[2])
    assert np.array_equal(y[6], x[6])
    assert not np.allclose(y[3], x[3])
