"""Nucleus (top-p) adjusted verify: the oracle's top-p, pinned.

"Fast Inference from Transformers via Speculative Decoding", section "The
loop", on the distributions being already adjusted for the sampling method:
nucleus sampling zeroes the tail and renormalises, and the algorithm treats the
adjusted p and q as the distributions.  Reading: a row keeps the smallest set of
largest-logit entries whose probability reaches top_p, every entry equal to the
last one kept as well; top-k, when also given, applies first.

1. top_p = 1 is the plain round, output for output.
2. A worked row with probabilities (0.5, 0.3, 0.15, 0.05): top_p = 0.7 keeps
   the first two, renormalised to (0.625, 0.375); top_p = 0.85 keeps three.
3. The defining properties hold on random rows with ties, read back through
   p(x) at every token: the kept set is closed upwards in the logits, its
   unadjusted mass reaches top_p, dropping its smallest tie group falls below
   top_p, and the adjusted probabilities are the renormalised ones.
4. A tiny top_p keeps only the argmax: with drafts at the draft argmax the
   round equals greedy verify.
5. Exactness holds for the adjusted distributions (chi-square, acceptance
   sum min(p', q')).
"""
import numpy as np
import pytest

import oracle
from tests._helpers import chisq_pvalue


def _probs(z, T=1.0):
    s = z.astype(np.float64) * float(np.float32(1.0) / np.float32(T))
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _p_everywhere(zrow, top_p, top_k=0, T=1.0):
    """p'(v) for every v of one target row, read through the oracle's p(x~)."""
    V = zrow.shape[0]
    zt = np.repeat(zrow[None, None, :], V, axis=0).astype(np.float32)
    zt = np.concatenate([zt, zt], axis=1)  # [V, 2, V]: gamma = 1
    zd = zt[:, :1].copy()
    xt = np.arange(V, dtype=np.int32)[:, None]
    out = oracle.spec_verify(zt, zd, xt, temperature=T, top_p=top_p, top_k=top_k)
    return out["p"][:, 0]


def test_top_p_one_is_the_plain_round():
    rng = np.random.default_rng(1)
    zt = rng.normal(0, 2, (6, 4, 200)).astype(np.float32)
    zd = (zt[:, :3] + rng.normal(0, 1, (6, 3, 200))).astype(np.float32)
    xt = rng.integers(0, 200, (6, 3)).astype(np.int32)
    a = oracle.spec_verify(zt, zd, xt, temperature=0.8, seed=2, rnd=3)
    b = oracle.spec_verify(zt, zd, xt, temperature=0.8, seed=2, rnd=3, top_p=1.0)
    for key in ("tokens", "counts", "p", "q", "ratio", "u", "flags"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    assert np.all(np.isinf(b["nucleus_gap"]))


@pytest.mark.parametrize("top_p,expect", [(0.7, [0.625, 0.375, 0.0, 0.0]),
                                          (0.85, [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0.0]),
                                          (0.4, [1.0, 0.0, 0.0, 0.0]),
                                          (0.999, [0.5, 0.3, 0.15, 0.05])])
def test_worked_row(top_p, expect):
    z = np.log(np.array([0.5, 0.3, 0.15, 0.05]))
    got = _p_everywhere(z.astype(np.float32), top_p)
    np.testing.assert_allclose(got, expect, rtol=1e-6)


@pytest.mark.parametrize("top_p,top_k,ties,T", [(0.9, 0, False, 1.0), (0.5, 0, True, 1.0),
                                                (0.75, 0, False, 0.6), (0.95, 20, True, 1.2),
                                                (0.3, 0, True, 0.9)])
def test_defining_properties(top_p, top_k, ties, T):
    rng = np.random.default_rng(int(top_p * 100) + top_k)
    V = 64
    for rep in range(4):
        z = (rng.integers(-5, 6, V) * 0.5 if ties else rng.normal(0, 2, V)).astype(np.float32)
        got = _p_everywhere(z, top_p, top_k, T)
        base = z.astype(np.float64)
        if top_k:
            kth = np.sort(base)[::-1][top_k - 1]
            base = np.where(base >= kth, base, -np.inf)
        p = _probs(base, T)
        kept = got > 0
        assert kept.any()
        # closed upwards in the logits
        assert np.all(base[~kept] < base[kept].min())
        # reaches top_p, and not without its smallest tie group
        mass = p[kept].sum()
        assert mass >= top_p - 1e-12
        smallest = base[kept].min()
        assert p[kept & (base > smallest)].sum() < top_p + 1e-12
        # the adjusted probabilities are the renormalised ones
        np.testing.assert_allclose(got[kept], p[kept] / mass, rtol=1e-9)


def test_tiny_top_p_is_greedy_verify():
    rng = np.random.default_rng(7)
    B, g, V = 200, 4, 64
    zt = rng.normal(0, 1, (B, g + 1, V)).astype(np.float32)
    zd = (zt[:, :g] + rng.normal(0, 0.7, (B, g, V))).astype(np.float32)
    xt = zd.argmax(-1).astype(np.int32)
    s = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=11, rnd=4, top_p=1e-9)
    gr = oracle.spec_verify_greedy(zt, xt)
    np.testing.assert_array_equal(s["tokens"], gr["tokens"])
    np.testing.assert_array_equal(s["counts"], gr["counts"])


@pytest.mark.parametrize("top_p,seed", [(0.6, 31), (0.9, 32)])
def test_exactness_on_adjusted_distributions(top_p, seed):
    rng = np.random.default_rng(seed)
    V, n = 10, 200_000
    zt1 = rng.normal(0, 1.5, (1, 2, V)).astype(np.float32)
    zd1 = (zt1[:, :1] + rng.normal(0, 1.0, (1, 1, V))).astype(np.float32)
    p1 = _p_everywhere(zt1[0, 0], top_p)
    q1 = _p_everywhere(zd1[0, 0], top_p)
    zt = np.repeat(zt1, n, axis=0)
    zd = np.repeat(zd1, n, axis=0)
    xt = rng.choice(V, size=(n, 1), p=q1 / q1.sum()).astype(np.int32)
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=seed, rnd=0, top_p=top_p)
    obs = np.bincount(out["tokens"][:, 0], minlength=V)
    support = p1 > 0
    assert obs[~support].sum() == 0
    assert chisq_pvalue(obs[support], p1[support]) > 1e-3
    acc = np.minimum(p1, q1).sum()
    assert abs(np.mean(out["counts"] == 1) - acc) < 5 * np.sqrt(acc * (1 - acc) / n)


@pytest.mark.parametrize("p", [0.0, -0.1, 1.5, float("nan")])
def test_top_p_out_of_range_rejected(p):
    zt = np.zeros((1, 2, 4), np.float32)
    zd = np.zeros((1, 1, 4), np.float32)
    xt = np.zeros((1, 1), np.int32)
    with pytest.raises(ValueError):
        oracle.spec_verify(zt, zd, xt, top_p=p)
