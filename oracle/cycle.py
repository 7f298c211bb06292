"""Speculative-decoding cycle accounting (oracle; test infrastructure only).

"DFlash: Block Diffusion for Flash Speculative Decoding", section 3.4.1,
Equation 1: the per-token latency of speculative decoding is the cycle time
(drafting plus verification) divided by the expected number of tokens a cycle
commits, tau, and the speedup is the autoregressive per-token latency divided by
that.  tau counts the bonus token, so a cycle with gamma draft tokens commits
between 1 and gamma + 1 tokens.
"""


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
