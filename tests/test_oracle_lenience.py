"""Lenience l: the oracle's variant of the comparison, pinned.

"Fast Inference from Transformers via Speculative Decoding", the paragraph on
sharper distributions (Appendix A.5 as summarised there): q(x) is multiplied by
l before the comparison, which accepts more, and the round loses exactness; no
token is then emitted more than 1/l times as often as the target would emit it.
The page changes only the comparison, so the correction after a rejection stays
the residual max(0, p - q) of Algorithm 1.

1. l = 1 is the exact round, output for output.
2. The rational enumeration with lenience meets what the page and the algebra
   fix: the first emitted token's rate is at most p(x)/l, the first draft is
   accepted with probability sum_x min(q(x), p(x)/l), the emitted distribution
   is still a distribution, and for l < 1 with p != q it is no longer p.
3. The oracle's round with lenience reproduces that enumeration (chi-square)
   and its acceptance rate.
4. l outside (0, 1] is rejected.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import exact
from tests._helpers import chisq_pvalue, logits_from_probs, sample_rows
from tests.test_oracle_exact import _random_tables


def _first_accept(dist):
    """P(the first draft is accepted) = P(the round emits two or more tokens)."""
    return sum(w for s, w in dist.items() if len(s) >= 2)


def test_lenience_one_is_the_exact_round():
    rng = np.random.default_rng(31)
    B, g, V = 16, 4, 300
    zt = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
    zd = (zt[:, :g] + rng.normal(0, 1, (B, g, V))).astype(np.float32)
    xt = rng.integers(0, V, (B, g)).astype(np.int32)
    a = oracle.spec_verify(zt, zd, xt, temperature=0.9, seed=5, rnd=2)
    b = oracle.spec_verify(zt, zd, xt, temperature=0.9, seed=5, rnd=2, lenience=1.0)
    for k in ("tokens", "counts", "p", "q", "ratio", "u", "flags"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("l", [Fraction(1, 2), Fraction(1, 10), Fraction(3, 4)])
@pytest.mark.parametrize("V,gamma,seed", [(3, 1, 40), (4, 2, 41), (5, 3, 42)])
def test_enumeration_with_lenience(V, gamma, seed, l):
    rng = np.random.default_rng(seed)
    P, Q = _random_tables(rng, V, gamma, zero_frac=0.0)
    dist = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma, lenience=l)
    assert sum(dist.values()) == 1
    first = exact.conditional_next(dist, (), V)
    p0, q0 = P[()], Q[()]
    for y in range(V):
        assert first[y] <= p0[y] / l  # no token more than 1/l times its target rate
    assert _first_accept(dist) == sum(min(q0[x], p0[x] / l) for x in range(V))
    if p0 != q0:
        assert first != p0  # exactness is lost
    # and the exact round is recovered at l = 1
    exact1 = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma)
    assert exact.conditional_next(exact1, (), V) == p0


def test_enumeration_lenience_accepts_more():
    rng = np.random.default_rng(43)
    V, gamma = 6, 2
    P, Q = _random_tables(rng, V, gamma, zero_frac=0.0)
    acc = [_first_accept(exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma,
                                               lenience=l))
           for l in (Fraction(1), Fraction(1, 2), Fraction(1, 10))]
    assert acc[0] < acc[1] < acc[2] <= 1


@pytest.mark.parametrize("V,gamma,seed,l", [(3, 2, 51, 0.5), (4, 1, 52, 0.1), (5, 2, 53, 0.25)])
def test_oracle_montecarlo_matches_enumeration_with_lenience(V, gamma, seed, l):
    rng = np.random.default_rng(seed)
    P, Q = _random_tables(rng, V, gamma, zero_frac=0.0)
    lf = Fraction(l).limit_denominator(1000)
    dist = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma, lenience=lf)
    n = 200_000
    xt = np.zeros((n, gamma), np.int32)
    zt = np.empty((n, gamma + 1, V), np.float32)
    zd = np.empty((n, gamma, V), np.float32)
    for i in range(gamma + 1):
        prefixes = [tuple(r) for r in xt[:, :i]]
        uniq = sorted(set(prefixes))
        lookup = {pre: k for k, pre in enumerate(uniq)}
        sel = np.array([lookup[pre] for pre in prefixes])
        ptab = np.array([[float(x) for x in P[pre]] for pre in uniq])
        zt[:, i] = logits_from_probs(ptab)[sel]
        if i < gamma:
            qtab = np.array([[float(x) for x in Q[pre]] for pre in uniq])
            zd[:, i] = logits_from_probs(qtab)[sel]
            xt[:, i] = sample_rows(rng, qtab[sel])
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=seed, rnd=3, lenience=l)
    seqs = list(dist.keys())
    index = {s: k for k, s in enumerate(seqs)}
    obs = np.zeros(len(seqs))
    for b in range(n):
        k = out["counts"][b]
        obs[index[tuple(int(t) for t in out["tokens"][b, :k + 1])]] += 1
    assert chisq_pvalue(obs, [float(dist[s]) for s in seqs]) > 1e-3
    acc = float(_first_accept(dist))
    assert abs(np.mean(out["counts"] >= 1) - acc) <= 5 * np.sqrt(acc * (1 - acc) / n)
    # the ratio the oracle reports is p / (l q)
    np.testing.assert_allclose(out["ratio"], out["p"] / (l * out["q"]), rtol=1e-15)


@pytest.mark.parametrize("l", [0.0, -0.5, 1.5, float("nan"), float("inf")])
def test_lenience_out_of_range_rejected(l):
    zt = np.zeros((1, 2, 4), np.float32)
    zd = np.zeros((1, 1, 4), np.float32)
    xt = np.zeros((1, 1), np.int32)
    with pytest.raises(ValueError):
        oracle.spec_verify(zt, zd, xt, lenience=l)
