"""Speculative-decoding cycle accounting (oracle; test infrastructure only).

"DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.1,
Equation 1: the per-token latency of speculative decoding is the cycle time
(drafting plus verification) divided by the expected number of tokens a cycle
commits, tau, and the speedup is the autoregressive per-token latency divided by
that.  tau counts the bonus token, so a cycle with gamma draft tokens commits
between 1 and gamma + 1 tokens.

It also holds the steady state between cycles (`commit`): the accepted path
becomes drafter context (DFlash page, section 3.4.3; DDTree page, section 3.4.5).
"""
import numpy as np


def per_token_latency(t_draft: float, t_verify: float, tau: float) -> float:
    """L = (T_draft + T_verify) / tau (Equation 1, denominator)."""
    if tau <= 0:
        raise ValueError("tau must be positive")
    return (t_draft + t_verify) / tau


def speedup(l_target: float, l_spec: float) -> float:
    """eta = L_target / L (Equation 1)."""
    return l_target / l_spec


def tau_of_cycle(accept_len: int) -> int:
    """Tokens committed by one cycle: the accepted draft tokens plus the bonus."""
    return accept_len + 1


def tau_bounds(gamma: int):
    """The range tau can take with gamma draft tokens per cycle: [1, gamma + 1]."""
    return 1, gamma + 1


def commit(accept_len, accepted, bonus, ctx_len, tree_feats):
    """Steady-state bookkeeping after one verified cycle (DFlash page, section
    3.4.3: verified tokens enter the drafter's cache as context, the cache is
    reused across cycles; DDTree page, section 3.4.5: only the accepted path
    stays).

    Per request r with a = accept_len[r]: the accepted path is node 0 (the
    cycle's anchor) followed by accepted[r][:a]; it occupies positions
    ctx_len[r] .. ctx_len[r] + a, so the next injection takes its a + 1 feature
    rows (tree_feats[r][node]) at pos0[r] = ctx_len[r]; then the context grows
    by a + 1 and the bonus token becomes the next anchor.

    Returns (row_off [n_req+1], pos0 [n_req], feats [sum of a+1, feat_dim],
    new ctx_len [n_req], new anchor [n_req]).
    """
    n_req = len(accept_len)
    row_off = [0]
    pos0, rows, new_ctx, new_anchor = [], [], [], []
    for r in range(n_req):
        a = int(accept_len[r])
        path = [0] + [int(x) for x in accepted[r][:a]]
        for node in path:
            rows.append(np.asarray(tree_feats[r][node]))
        row_off.append(row_off[-1] + len(path))
        pos0.append(int(ctx_len[r]))
        new_ctx.append(int(ctx_len[r]) + a + 1)
        new_anchor.append(int(bonus[r]))
    return (np.array(row_off), np.array(pos0), np.stack(rows), np.array(new_ctx),
            np.array(new_anchor))
