"""Pins for the cycle accounting (Equation 1 of the DFlash page) against the
numbers the pages print, and for the steady-state commit (a hand example and
its agreement with the walk's tau over several cycles)."""
import json
import os

import numpy as np
import pytest

from oracle import cycle
from oracle import cycle as oc


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_eq1_worked_example(golden_dir):
    g = _load(golden_dir, "eq1_worked_example.json")
    L = cycle.per_token_latency(g["t_draft_ms"], g["t_verify_ms"], g["tau"])
    assert L == pytest.approx(g["per_token_latency_ms"], rel=1e-12)
    assert cycle.speedup(g["l_target_ms"], L) == pytest.approx(g["speedup"], rel=1e-12)


def test_a100_cycle_identity(golden_dir):
    g = _load(golden_dir, "a100_cycle.json")
    # the cycle is drafting plus verification; tau = 1 turns it into a per-token cost
    assert cycle.per_token_latency(g["t_draft_ms"], g["t_verify_ms"], 1) == \
        pytest.approx(g["cycle_ms"], rel=1e-12)
    # a cycle committing only the bonus token is slower than plain decoding
    # (the explainer's remark that tau = 1 loses to not speculating)
    L1 = cycle.per_token_latency(g["t_draft_ms"], g["t_verify_ms"], 1)
    assert cycle.speedup(g["target_pass_ms"], L1) < 1.0
    # and tau = 2 is already a win on these numbers
    assert cycle.speedup(g["target_pass_ms"],
                         cycle.per_token_latency(g["t_draft_ms"], g["t_verify_ms"], 2)) > 1.0


def test_tau_bounds_include_bonus():
    # gamma draft tokens: all rejected -> 1 (bonus only); all accepted -> gamma + 1
    assert cycle.tau_bounds(16) == (1, 17)
    assert cycle.tau_of_cycle(0) == 1
    assert cycle.tau_of_cycle(16) == 17


def test_rejects_nonpositive_tau():
    with pytest.raises(ValueError):
        cycle.per_token_latency(1.0, 1.0, 0)


def test_commit_hand_example():
    # request 0 accepts nodes 3 then 7 (tau = 3), request 1 accepts nothing
    # (tau = 1: only its anchor becomes context)
    feats = np.arange(2 * 9 * 2, dtype=np.float64).reshape(2, 9, 2)
    accepted = np.array([[3, 7, -1], [-1, -1, -1]])
    row_off, pos0, rows, ctx, anchor = oc.commit([2, 0], accepted, [55, 66], [100, 40], feats)
    assert list(row_off) == [0, 3, 4]
    assert list(pos0) == [100, 40]
    assert list(ctx) == [103, 41]
    assert list(anchor) == [55, 66]
    assert np.array_equal(rows, np.stack([feats[0][0], feats[0][3], feats[0][7], feats[1][0]]))


def test_commit_matches_the_walk_and_eq1_tau():
    # the context grows by tau = accept_len + 1 per cycle, the count Equation 1
    # divides by; over several cycles ctx_len advances by the sum of the taus
    from oracle import ddtree as odt
    rng = np.random.default_rng(3)
    ctx = np.array([10, 20])
    total = np.zeros(2, dtype=int)
    for cyc in range(4):
        lp = np.sort(rng.normal(size=(2, 4, 3)).astype(np.float32) - 3, axis=2)[:, :, ::-1]
        ids = np.stack([[rng.choice(50, 3, replace=False) for _ in range(4)] for _ in range(2)])
        trees = [odt.build_tree(np.ascontiguousarray(lp[r]), ids[r].astype(np.int32), 1, 8)
                 for r in range(2)]
        al, acc, bon = [], [], []
        for r, t in enumerate(trees):
            target = np.full(9, -1)
            if t["n_nodes"] >= 1:
                target[0] = t["tok"][1]          # the walk takes node 1, then stops
            a, nodes, b = odt.accept_walk(t["tok"], t["parent"], t["n_nodes"], target, 4)
            al.append(a)
            acc.append(nodes)
            bon.append(b)
        feats = rng.normal(size=(2, 9, 4))
        row_off, pos0, rows, ctx2, _ = oc.commit(al, acc, bon, ctx, feats)
        assert list(pos0) == list(ctx)
        assert list(ctx2 - ctx) == [oc.tau_of_cycle(a) for a in al]
        assert row_off[-1] == rows.shape[0] == sum(a + 1 for a in al)
        total += ctx2 - ctx
        ctx = ctx2
    assert list(ctx) == list(np.array([10, 20]) + total)


def test_steady_state_cycles_equal_one_injection_of_the_history():
    # Several oracle cycles at the tiny fp32 shape (inject the previous accepted
    # path, draft, top-K, tree, walk against a first-child target, commit).  The
    # cache they leave must equal one injection of the whole accepted history at
    # its positions, and the next block's logits must agree: a wrong pos0, an
    # off-by-one in tau or a path row out of order fails one of the two.
    from block_diffusion_speculative_kv_gb300 import synth
    from block_diffusion_speculative_kv_gb300.configs import TINY_DRAFTER
    from oracle import ddtree as odt
    from oracle import drafter as od
    s = TINY_DRAFTER
    L, K, B, D = 8, 3, 12, 7
    w = synth.drafter_weights(s, 3)
    ow = {k: ([od.f64(t) for t in v] if isinstance(v, list) else od.f64(v)) for k, v in w.items()}
    dims = dict(n_layers=s.n_layers, d=s.d, n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim,
                vocab=s.vocab, mask_id=s.mask_id, rope_theta=s.rope_theta, rms_eps=s.rms_eps)
    cap, ctx = 64, 10
    fd = s.n_feat * s.d_feat
    rng = np.random.default_rng(9)
    ck = [np.zeros((s.n_kv, cap, s.head_dim)) for _ in range(s.n_layers)]
    cv = [np.zeros((s.n_kv, cap, s.head_dim)) for _ in range(s.n_layers)]

    def inject(rows, pos):
        f = od.fuse_features(rows, ow["w_proj"])
        for l in range(s.n_layers):
            k_, v_ = od.inject_kv(f, ow["uk"][l], ow["uv"][l], pos, s.n_kv, s.head_dim,
                                  s.rope_theta)
            ck[l][:, pos] = k_
            cv[l][:, pos] = v_

    history = [rng.normal(size=(ctx, fd))]
    inject(history[0], np.arange(ctx))
    anchor, pending, pos0 = 5, None, None
    taus = []
    for cyc in range(4):
        if pending is not None:
            inject(pending, pos0 + np.arange(len(pending)))
        logits = od.drafter_block(ow, dims, ck, cv, ctx, anchor, L)
        ids, lp, _ = od.logits_topk(logits, K)
        t = odt.build_tree(lp.astype(np.float32), ids.astype(np.int32), anchor, B)
        target = np.full(B + 1, (anchor + 1) % s.vocab)
        for i in range(t["n_nodes"] + 1):      # agree with the first child, except at odd tokens
            ch = [c for c in range(1, t["n_nodes"] + 1) if t["parent"][c] == i]
            if ch and t["tok"][ch[0]] % 2 == 0:
                target[i] = t["tok"][ch[0]]
        a, acc, bonus = odt.accept_walk(t["tok"], t["parent"], t["n_nodes"], target, D)
        tree_feats = rng.normal(size=(1, B + 1, fd))
        row_off, p0, rows, ctx2, anchor2 = oc.commit([a], [acc], [bonus], [ctx], tree_feats)
        assert row_off[-1] == a + 1 and p0[0] == ctx and ctx2[0] == ctx + a + 1
        history.append(rows)
        pending, pos0, ctx, anchor = rows, int(p0[0]), int(ctx2[0]), int(anchor2[0])
        taus.append(a + 1)
    inject(pending, pos0 + np.arange(len(pending)))
    # one injection of the whole history into a fresh cache
    full = np.concatenate(history)
    assert full.shape[0] == ctx == 10 + sum(taus)
    ck_ref = [np.zeros_like(c) for c in ck]
    cv_ref = [np.zeros_like(c) for c in cv]
    f = od.fuse_features(full, ow["w_proj"])
    for l in range(s.n_layers):
        k_, v_ = od.inject_kv(f, ow["uk"][l], ow["uv"][l], np.arange(ctx), s.n_kv, s.head_dim,
                              s.rope_theta)
        ck_ref[l][:, :ctx] = k_
        cv_ref[l][:, :ctx] = v_
        assert np.allclose(ck[l], ck_ref[l], atol=1e-12) and np.allclose(cv[l], cv_ref[l], atol=1e-12)
    a1 = od.drafter_block(ow, dims, ck, cv, ctx, anchor, L)
    a2 = od.drafter_block(ow, dims, ck_ref, cv_ref, ctx, anchor, L)
    assert np.allclose(a1, a2, atol=1e-12)
    assert max(taus) > 1      # some cycle accepted a draft token
