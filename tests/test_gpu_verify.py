"""GPU parity of the verification-side tree attention and the depth position
ids (DDTree page, 3.4.5) against the oracle, through the C ABI.

Tolerance: attention outputs are bf16 and the scores run through bf16
probabilities, so per (node, head) row max|out_gpu - out_ora| <= 2e-2 *
max|out_ora| (the bar used for the drafter's bf16 logits); rotated rows within
1e-2 of the oracle per row (bf16 in and out).  Rows past the last node must be
exactly zero."""
import math

import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd
from oracle import ddtree as odt
from oracle import verify as ov

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bf(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(DEV)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _tree(seed, B, D, K):
    rng = np.random.default_rng(seed)
    raw = rng.normal(size=(D, K + 3)) * 1.5
    m = raw.max(1, keepdims=True)
    lp = raw - (m + np.log(np.exp(raw - m).sum(1, keepdims=True)))
    lp = -np.sort(-lp, axis=1)[:, :K].astype(np.float32)
    ids = np.stack([rng.choice(1000, size=K, replace=False) for _ in range(D)]).astype(np.int32)
    t = odt.build_tree(lp, ids, 7, B)
    return t


def _case(seed, n_req, n_q, n_kv, B, ctxs, cap, D=8, K=4, scale=0.35):
    hd = 128
    rng = np.random.default_rng(seed)
    trees = [_tree(seed * 10 + r, B, D, K) for r in range(n_req)]
    n_nodes = np.array([t["n_nodes"] for t in trees], dtype=np.int32)
    mask = np.stack([t["mask"] for t in trees]).astype(np.uint32)
    depth = np.stack([t["depth"] for t in trees]).astype(np.int32)
    q = _bf(rng.normal(size=(n_req, B + 1, n_q * hd)) * scale)
    k = _bf(rng.normal(size=(n_req, B + 1, n_kv * hd)) * scale)
    v = _bf(rng.normal(size=(n_req, B + 1, n_kv * hd)))
    ck = _bf(rng.normal(size=(n_req, n_kv, cap, hd)) * scale)
    cv = _bf(rng.normal(size=(n_req, n_kv, cap, hd)))
    d = dict(q=q, k=k, v=v, ck=ck, cv=cv, n_nodes=n_nodes, mask=mask, depth=depth,
             ctx=np.asarray(ctxs, dtype=np.int32), n_q=n_q, n_kv=n_kv, B=B, hd=hd)
    return d


def _run(d):
    n_req = d["q"].shape[0]
    out = torch.full_like(d["q"], 7.0)   # stale values must be overwritten
    ws = torch.zeros(bd.tree_attention_workspace_bytes(n_req, d["n_q"], d["n_kv"], d["hd"],
                                                       d["B"], int(d["ctx"].max())),
                     dtype=torch.uint8, device=DEV)
    mask = torch.as_tensor(d["mask"].view(np.int32), device=DEV)
    bd.tree_attention(d["q"], d["k"], d["v"], d["ck"], d["cv"],
                      torch.as_tensor(d["ctx"], device=DEV), int(d["ctx"].max()), mask,
                      torch.as_tensor(d["n_nodes"], device=DEV), out, ws)
    torch.cuda.synchronize()
    return out


def _oracle_row(d, r, i, h):
    hd, n_q, n_kv = d["hd"], d["n_q"], d["n_kv"]
    g = h // (n_q // n_kv)
    ctx = int(d["ctx"][r])
    anc = ov.ancestors(d["mask"][r, i], d["B"] + 1)
    q = _f64(d["q"][r, i, h * hd:(h + 1) * hd])
    keys = np.concatenate([_f64(d["ck"][r, g, :ctx]),
                           _f64(d["k"][r, anc][:, g * hd:(g + 1) * hd])])
    vals = np.concatenate([_f64(d["cv"][r, g, :ctx]),
                           _f64(d["v"][r, anc][:, g * hd:(g + 1) * hd])])
    s = keys @ q / math.sqrt(hd)
    p = np.exp(s - s.max())
    return (p / p.sum()) @ vals


def _check_rows(d, out, rows):
    hd = d["hd"]
    for r, i, h in rows:
        ref = _oracle_row(d, r, i, h)
        got = _f64(out[r, i, h * hd:(h + 1) * hd])
        err = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-6)
        assert err <= 2e-2, (r, i, h, float(err))


def test_tree_attention_small_full():
    d = _case(1, n_req=2, n_q=8, n_kv=2, B=40, ctxs=[300, 0], cap=320)
    out = _run(d)
    full = ov.tree_attention  # the oracle's own all-rows form agrees with the per-row one
    for r in range(2):
        ref = full(_f64(d["q"][r]).reshape(41, 8, 128), _f64(d["k"][r]).reshape(41, 2, 128),
                   _f64(d["v"][r]).reshape(41, 2, 128), _f64(d["ck"][r]), _f64(d["cv"][r]),
                   int(d["ctx"][r]), d["mask"][r], int(d["n_nodes"][r]), 8, 2)
        got = _f64(out[r]).reshape(41, 8, 128)
        for i in range(int(d["n_nodes"][r]) + 1):
            for h in range(8):
                err = np.max(np.abs(got[i, h] - ref[i, h])) / np.max(np.abs(ref[i, h]))
                assert err <= 2e-2, (r, i, h, float(err))
        assert torch.count_nonzero(out[r, int(d["n_nodes"][r]) + 1:]) == 0


def test_tree_attention_ragged_tiles_and_dead_rows():
    # 64 + 1 rows (a partial last query tile), small trees (many dead rows),
    # contexts that end inside a key tile and a context of one slot
    d = _case(2, n_req=3, n_q=4, n_kv=1, B=64, ctxs=[1, 777, 1030], cap=1100, D=3, K=3)
    out = _run(d)
    rows = []
    for r in range(3):
        nn = int(d["n_nodes"][r])
        for i in sorted({0, 1, nn // 2, nn}):
            for h in (0, 3):
                rows.append((r, i, h))
        assert torch.count_nonzero(out[r, nn + 1:]) == 0
    _check_rows(d, out, rows)


def test_tree_attention_target_shape_sampled():
    # a Qwen3-8B-shaped target layer: 32/8 heads of 128, 8192 context slots,
    # a 256-node tree; rows sampled across query tiles and heads
    d = _case(3, n_req=1, n_q=32, n_kv=8, B=256, ctxs=[8192], cap=8192, D=15, K=8)
    out = _run(d)
    nn = int(d["n_nodes"][0])
    rng = np.random.default_rng(0)
    nodes = sorted(set([0, 1, 15, 16, 17, nn] + list(rng.integers(0, nn + 1, size=10))))
    rows = [(0, int(i), int(h)) for i in nodes for h in (0, 5, 31)]
    _check_rows(d, out, rows)


def test_tree_attention_target_shape_full_heads():
    # every node of two heads at the Qwen3-8B target shape: all nine query
    # tiles (the last holds one node), both context chunks and the tree keys
    d = _case(5, n_req=1, n_q=32, n_kv=8, B=256, ctxs=[8192], cap=8192, D=15, K=8)
    out = _run(d)
    nn = int(d["n_nodes"][0])
    _check_rows(d, out, [(0, i, h) for i in range(nn + 1) for h in (7, 28)])
    assert torch.count_nonzero(out[0, nn + 1:]) == 0


def test_tree_attention_two_heads_per_group_nan_past_context():
    # G = 2 (rows 64..127 of each tile unused); cache slots past each request's
    # context hold NaN: masked scores and zeroed value rows keep them out
    d = _case(6, n_req=2, n_q=16, n_kv=8, B=100, ctxs=[500, 1061], cap=1200, D=6, K=5)
    for r, c in enumerate(d["ctx"]):
        d["ck"][r, :, int(c):] = float("nan")
        d["cv"][r, :, int(c):] = float("nan")
    out = _run(d)
    assert torch.isfinite(out.float()).all()
    rows = []
    for r in range(2):
        nn = int(d["n_nodes"][r])
        rows += [(r, i, h) for i in sorted({0, 1, 31, 32, nn}) if i <= nn for h in (0, 3, 15)]
        assert torch.count_nonzero(out[r, nn + 1:]) == 0
    _check_rows(d, out, rows)


def test_tree_attention_large_tree():
    # B = 1024: 1025 nodes, 33 mask words per row, up to nine tiles of tree keys
    d = _case(7, n_req=1, n_q=8, n_kv=2, B=1024, ctxs=[300], cap=384, D=16, K=8)
    out = _run(d)
    nn = int(d["n_nodes"][0])
    rng = np.random.default_rng(1)
    nodes = sorted(set([0, 1, 127, 128, 1000, nn] + list(rng.integers(0, nn + 1, size=12))))
    _check_rows(d, out, [(0, int(i), h) for i in nodes if i <= nn for h in (0, 7)])


def test_tree_attention_root_only():
    d = _case(8, n_req=1, n_q=4, n_kv=1, B=0, ctxs=[129], cap=256)
    out = _run(d)
    _check_rows(d, out, [(0, 0, h) for h in range(4)])


def test_tree_rope_matches_oracle():
    rng = np.random.default_rng(4)
    n_req, B, heads, hd, theta = 2, 30, 3, 128, 1e6
    trees = [_tree(40 + r, B, 6, 3) for r in range(n_req)]
    depth = np.stack([t["depth"] for t in trees]).astype(np.int32)
    ctx = np.array([100, 4097], dtype=np.int32)
    ld = heads * hd + 64          # a padded row
    x = _bf(rng.normal(size=(n_req, B + 1, ld)))
    before = x.clone()
    bd.tree_rope(x, heads, hd, theta, torch.as_tensor(ctx, device=DEV),
                 torch.as_tensor(depth, device=DEV))
    torch.cuda.synchronize()
    for r in range(n_req):
        ref = ov.tree_rope(_f64(before[r, :, :heads * hd]).reshape(B + 1, heads, hd), int(ctx[r]),
                           depth[r], theta)
        got = _f64(x[r, :, :heads * hd]).reshape(B + 1, heads, hd)
        err = np.max(np.abs(got - ref), axis=2) / np.max(np.abs(ref), axis=2)
        assert np.all(err <= 1e-2), float(err.max())
        # the padding columns are untouched
        assert torch.equal(x[r, :, heads * hd:], before[r, :, heads * hd:])
