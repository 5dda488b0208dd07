"""Closed forms of the pages' analysis (test infrastructure, used by the oracle's pins).

Each function cites the page and the statement it restates.  The pages print
numeric values for all of them; ``tests/test_oracle_theory.py`` pins each
function to those values before any other test uses it.
"""
from __future__ import annotations


def expected_tokens(alpha: float, gamma: int) -> float:
    """Expected tokens per round with i.i.d. acceptance alpha and draft length gamma.

    "Speculative Decoding" (course notes), Proposition "Expected tokens per
    verification round"; "Fast Inference from Transformers via Speculative
    Decoding", section "Tokens per target run, equation (1)".
    """
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def tokens_histogram(alpha: float, gamma: int) -> list[float]:
    """P(a round emits k tokens), k = 1..gamma+1.

    "Fast Inference from Transformers via Speculative Decoding", section
    "Tokens per target run, equation (1)", the Figure 4 paragraph:
    alpha^(k-1) (1-alpha) for k <= gamma and alpha^gamma for the clean sweep.
    """
    h = [alpha ** (k - 1) * (1.0 - alpha) for k in range(1, gamma + 1)]
    h.append(alpha ** gamma)
    return h


def speedup(alpha: float, gamma: int, c: float) -> float:
    """Expected walltime improvement, Theorem 3.8 / equation (5).

    "Fast Inference from Transformers via Speculative Decoding", section
    "Walltime, the cost of the draft, and choosing gamma"; course notes,
    Corollary "Speedup and the optimal draft length".
    """
    return expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def ops_factor(alpha: float, gamma: int, c_hat: float) -> float:
    """Factor by which total arithmetic grows, Theorem 3.11.

    The display is lost in the page's text ("Walltime, the cost of the draft,
    and choosing gamma"); this is the reading that reproduces all three
    operation factors of its Table 1: each round scores gamma+1 target
    positions plus gamma draft runs of relative cost c_hat, and yields
    expected_tokens(alpha, gamma) tokens.
    """
    return (gamma * c_hat + gamma + 1.0) / expected_tokens(alpha, gamma)


def rejection_sampling_rate(p, q) -> float:
    """Acceptance rate 1/r_max of ordinary rejection sampling with proposal q.

    "Fast Inference from Transformers via Speculative Decoding", section
    "Speculative sampling: the accept/reject rule" (Appendix A.2 comparison).
    """
    r_max = max(pi / qi for pi, qi in zip(p, q) if qi > 0)
    return 1.0 / r_max
