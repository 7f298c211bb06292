"""Pins for the cycle accounting (Equation 1 of the DFlash page) against the
numbers the pages print."""
import json
import os

import pytest

from oracle import cycle


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
