"""Exact enumeration of one verify round over rational distributions.

Test infrastructure (part of the oracle).  For small V and gamma it sums the
probability of every branch of the round analytically, in exact rational
arithmetic (``fractions.Fraction``), following the steps of Algorithm 1
("Fast Inference from Transformers via Speculative Decoding", section "The
loop: draft, verify in one pass, keep a prefix") and of the course notes'
algorithm box ("Speculative Decoding", "The algorithm"):

  draft x_i ~ q_i(. | prefix), accept w.p. min(1, p_i(x_i)/q_i(x_i)),
  on the first rejection emit y ~ max(0, p_i - q_i) / sum, after gamma
  acceptances emit y ~ p_gamma(. | prefix).

The distributions may depend on the drafted prefix (a tiny autoregressive
"model"): ``p_of(prefix)`` and ``q_of(prefix)`` return lists of Fractions.
"""
from __future__ import annotations

from fractions import Fraction
from typing import Callable, Dict, Sequence, Tuple

Dist = Sequence[Fraction]


def residual(p: Dist, q: Dist):
    """max(0, p - q) normalised; None when it has no mass.

    Same page, "Speculative sampling: the accept/reject rule", residual (2).
    """
    r = [max(pi - qi, Fraction(0)) for pi, qi in zip(p, q)]
    s = sum(r)
    if s == 0:
        return None
    return [ri / s for ri in r]


def enumerate_round(p_of: Callable[[Tuple[int, ...]], Dist],
                    q_of: Callable[[Tuple[int, ...]], Dist],
                    V: int, gamma: int, lenience: Fraction = Fraction(1)
                    ) -> Dict[Tuple[int, ...], Fraction]:
    """Exact distribution of the emitted token tuple of one round.

    lenience l: the comparison uses l q(x), i.e. accept w.p. min(1, p/(l q))
    (same page, the paragraph on sharper distributions: Appendix A.5); the
    correction after a rejection is the residual above, unchanged."""
    out: Dict[Tuple[int, ...], Fraction] = {}

    def add(seq, w):
        out[seq] = out.get(seq, Fraction(0)) + w

    def walk(prefix: Tuple[int, ...], w: Fraction):
        i = len(prefix)
        p = p_of(prefix)
        if i == gamma:  # every draft accepted: bonus token from p_gamma
            for y in range(V):
                if p[y]:
                    add(prefix + (y,), w * p[y])
            return
        q = q_of(prefix)
        res = residual(p, q)
        for x in range(V):
            if q[x] == 0:
                continue
            a = min(Fraction(1), p[x] / (lenience * q[x]))
            if a:
                walk(prefix + (x,), w * q[x] * a)
            rej = w * q[x] * (1 - a)
            if rej:
                # a rejection is only possible when p != q, so res is not None
                for y in range(V):
                    if res[y]:
                        add(prefix + (y,), rej * res[y])

    walk((), Fraction(1))
    return out


def conditional_next(dist: Dict[Tuple[int, ...], Fraction], prefix: Tuple[int, ...], V: int):
    """P(out_j = y | out[:j] = prefix, round emitted more than j tokens), j = len(prefix).

    Returns None when the conditioning event has probability zero.
    """
    j = len(prefix)
    num = [Fraction(0)] * V
    for seq, w in dist.items():
        if len(seq) > j and seq[:j] == prefix:
            num[seq[j]] += w
    den = sum(num)
    if den == 0:
        return None
    return [x / den for x in num]
