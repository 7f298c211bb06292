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
