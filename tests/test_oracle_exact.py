"""Exhaustive enumeration pins (V <= 8, gamma <= 3).

1. The exact branch-probability enumeration satisfies the exactness theorem
   ("Speculative Decoding" course notes, 'Exactness'; 'Fast Inference ...',
   Appendix A.1): given that a round reached position j with the drafted
   prefix y_<j, the token it emits at j is distributed exactly as
   p_j(. | y_<j), in rational arithmetic, for prefix-dependent tables.
2. The oracle's Monte Carlo verify reproduces the enumerated distribution of
   whole output tuples (chi-square).
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import exact
from tests._helpers import chisq_pvalue, logits_from_probs, sample_rows


def _random_tables(rng, V, gamma, zero_frac=0.2):
    """Prefix-dependent rational distributions (a tiny autoregressive model).

    Some entries are zero (tokens one model never proposes), but every
    distribution keeps at least two tokens so the round has several outcomes."""
    def rand_dist(allow_zero):
        w = [int(x) for x in rng.integers(1, 9, V)]
        if allow_zero:
            for j in range(V):
                if rng.random() < zero_frac:
                    w[j] = 0
            while sum(1 for x in w if x) < min(2, V):
                w[int(rng.integers(0, V))] = int(rng.integers(1, 9))
        s = sum(w)
        return [Fraction(x, s) for x in w]

    P, Q = {}, {}
    for L in range(gamma + 1):
        for pre in itertools.product(range(V), repeat=L):
            P[pre] = rand_dist(allow_zero=True)
            if L < gamma:
                Q[pre] = rand_dist(allow_zero=True)
    return P, Q


@pytest.mark.parametrize("V,gamma,seed", [(2, 1, 0), (3, 2, 1), (4, 3, 2), (5, 2, 3), (8, 1, 4),
                                          (8, 2, 5), (3, 3, 6)])
def test_enumeration_is_exact(V, gamma, seed):
    rng = np.random.default_rng(seed)
    P, Q = _random_tables(rng, V, gamma)
    dist = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma)
    assert sum(dist.values()) == 1
    assert all(1 <= len(s) <= gamma + 1 for s in dist)
    for j in range(gamma + 1):
        for pre in itertools.product(range(V), repeat=j):
            cond = exact.conditional_next(dist, pre, V)
            if cond is not None:
                assert cond == P[pre], (j, pre)
    # first emitted token is exactly p_0
    assert exact.conditional_next(dist, (), V) == P[()]


def test_invariant_catches_a_planted_mistake(monkeypatch):
    """The pin has teeth: resampling from p itself after a rejection (instead of
    the residual max(0, p-q)) breaks the exactness invariant."""
    rng = np.random.default_rng(9)
    V, gamma = 3, 1
    P, Q = _random_tables(rng, V, gamma, zero_frac=0.0)
    good = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma)
    assert exact.conditional_next(good, (), V) == P[()]
    monkeypatch.setattr(exact, "residual", lambda p, q: list(p))
    bad = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma)
    assert exact.conditional_next(bad, (), V) != P[()]


@pytest.mark.parametrize("V,gamma,seed", [(3, 2, 11), (4, 3, 12), (8, 1, 13)])
def test_oracle_montecarlo_matches_enumeration(V, gamma, seed):
    rng = np.random.default_rng(seed)
    P, Q = _random_tables(rng, V, gamma)
    dist = exact.enumerate_round(P.__getitem__, Q.__getitem__, V, gamma)
    n = 200_000
    # draw each trial's drafts autoregressively from q(. | prefix)
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
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=seed, rnd=1)
    seqs = list(dist.keys())
    index = {s: k for k, s in enumerate(seqs)}
    obs = np.zeros(len(seqs))
    for b in range(n):
        k = out["counts"][b]
        obs[index[tuple(int(t) for t in out["tokens"][b, :k + 1])]] += 1
    assert chisq_pvalue(obs, [float(dist[s]) for s in seqs]) > 1e-3
