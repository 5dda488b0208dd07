"""Draft sampling x ~ q (the draft side of a round), pinned.

"Fast Inference from Transformers via Speculative Decoding", section "The
loop", step 1: the draft model runs gamma times and each draft token is drawn
from its distribution q_i; the course notes' "The algorithm" states the same
x_{t+i} ~ q(. | prefix).  The oracle draws it as a Gumbel-max over the
temperature-scaled logits with its own Philox stream (tag 2).

1. Over many rounds the drawn tokens follow softmax(z / T) (chi-square), for
   several temperatures and rows with -inf entries.
2. A tiny temperature draws the argmax.
3. lse is scipy's logsumexp of the scaled logits and q(x) = exp(s_x - lse).
4. An all -inf row draws token 0 with q = 0.
"""
import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from tests._helpers import chisq_pvalue


@pytest.mark.parametrize("T,seed", [(1.0, 1), (0.6, 2), (1.7, 3)])
def test_draws_follow_the_softmax(T, seed):
    rng = np.random.default_rng(seed)
    V, n = 8, 40_000
    z = rng.normal(0, 1.5, V).astype(np.float32)
    z[5] = -np.inf
    inv_t = float(np.float32(1.0) / np.float32(T))
    p = np.exp(z.astype(np.float64) * inv_t - logsumexp(z.astype(np.float64) * inv_t))
    # one batch row per trial: rows differ in b, so every trial has its own noise
    out = oracle.draft_sample(np.tile(z, (n, 1)), temperature=T, seed=seed, rnd=7, pos=2)
    obs = np.bincount(out["tokens"], minlength=V)
    assert obs[5] == 0
    keep = p > 0
    assert chisq_pvalue(obs[keep], p[keep]) > 1e-3
    # and across rounds for one batch row
    toks = np.array([oracle.draft_sample(z[None], temperature=T, seed=seed, rnd=r,
                                         pos=0)["tokens"][0] for r in range(6000)])
    assert chisq_pvalue(np.bincount(toks, minlength=V)[keep], p[keep]) > 1e-3


def test_tiny_temperature_draws_the_argmax():
    rng = np.random.default_rng(4)
    z = rng.normal(0, 1, (50, 300)).astype(np.float32)
    out = oracle.draft_sample(z, temperature=1e-4, seed=3, rnd=1, pos=1)
    np.testing.assert_array_equal(out["tokens"], z.argmax(1))


def test_lse_and_q_match_scipy():
    rng = np.random.default_rng(5)
    z = rng.normal(0, 3, (20, 1000)).astype(np.float32)
    T = 0.8
    inv_t = float(np.float32(1.0) / np.float32(T))
    out = oracle.draft_sample(z, temperature=T, seed=9, rnd=0, pos=3)
    s = z.astype(np.float64) * inv_t
    lse = logsumexp(s, axis=1)
    np.testing.assert_allclose(out["lse"], lse, rtol=1e-13)
    q = np.exp(s[np.arange(20), out["tokens"]] - lse)
    np.testing.assert_allclose(out["q"], q, rtol=1e-12)


def test_empty_row():
    z = np.full((2, 16), -np.inf, np.float32)
    z[1, 3] = 0.0
    out = oracle.draft_sample(z, temperature=1.0, seed=0, rnd=0, pos=0)
    assert out["tokens"][0] == 0 and out["q"][0] == 0.0
    assert out["tokens"][1] == 3 and out["q"][1] == 1.0
