"""Planted mistakes: each test puts a plausible error into the oracle (on the
CPU, through monkeypatch, undone afterwards) and checks that the pin meant to
catch it fails.  A pin that still passed with the mistake in place would not
be pinning anything."""
import importlib

import numpy as np
import pytest

from oracle import cycle as oc
from oracle import drafter as od
from oracle import sampling as osm
from oracle import verify as ov


def _pin(module, name):
    return getattr(importlib.import_module(module), name)


def test_gumbel_sign_flip_is_caught(monkeypatch):
    monkeypatch.setattr(osm, "gumbel", lambda u: np.log(-np.log(np.asarray(u, np.float32))))
    with pytest.raises(AssertionError):
        _pin("test_oracle_sampling", "test_gumbel_max_draws_follow_softmax")()


def test_wrong_generator_increment_is_caught(monkeypatch):
    monkeypatch.setattr(osm, "GAMMA", 0x9E3779B97F4A7C13)
    with pytest.raises(AssertionError):
        _pin("test_oracle_sampling", "test_splitmix64_published_outputs")()


def test_chain_rank_zero_is_caught(monkeypatch):
    real = osm.chain_tree

    def rank_zero(root_tok, tokens, B):
        t = real(root_tok, tokens, B)
        t["rank"] = np.where(t["rank"] > 0, 0, t["rank"])
        return t
    monkeypatch.setattr(osm, "chain_tree", rank_zero)
    with pytest.raises(AssertionError):
        _pin("test_oracle_sampling", "test_chain_tree_mask_and_walk")()


def test_commit_off_by_one_position_is_caught(monkeypatch):
    real = oc.commit

    def shifted(*a, **k):
        row_off, pos0, rows, ctx, anchor = real(*a, **k)
        return row_off, pos0 + 1, rows, ctx + 1, anchor
    monkeypatch.setattr(oc, "commit", shifted)
    with pytest.raises(AssertionError):
        _pin("test_oracle_cycle", "test_steady_state_cycles_equal_one_injection_of_the_history")()


def test_commit_reversed_path_is_caught(monkeypatch):
    real = oc.commit

    def reversed_rows(accept_len, accepted, bonus, ctx_len, tree_feats):
        row_off, pos0, rows, ctx, anchor = real(accept_len, accepted, bonus, ctx_len, tree_feats)
        for r in range(len(accept_len)):
            rows[row_off[r]:row_off[r + 1]] = rows[row_off[r]:row_off[r + 1]][::-1].copy()
        return row_off, pos0, rows, ctx, anchor
    monkeypatch.setattr(oc, "commit", reversed_rows)
    with pytest.raises(AssertionError):
        _pin("test_oracle_cycle", "test_commit_hand_example")()


def test_tree_attention_ignoring_the_mask_is_caught(monkeypatch):
    monkeypatch.setattr(ov, "ancestors", lambda mask_row, width: np.arange(width))
    with pytest.raises(AssertionError):
        _pin("test_oracle_verify", "test_star_branches_see_only_root_and_themselves")()


def test_rope_rotation_direction_is_caught(monkeypatch):
    real = od.apply_rope
    monkeypatch.setattr(od, "apply_rope", lambda x, pos, theta: real(x, -np.asarray(pos), theta))
    with pytest.raises(AssertionError):
        _pin("test_oracle_drafter", "test_rope_matches_complex_rotation")()
