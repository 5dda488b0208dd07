"""Top-k adjusted verify: the oracle's top-k, pinned.

"Fast Inference from Transformers via Speculative Decoding", section "The
loop", on the distributions being already adjusted for the sampling method:
top-k zeroes the tail and renormalises, and the algorithm then treats the
adjusted p and q as the distributions.  Reading for the boundary: a row keeps
every entry whose (scaled) logit is at least its k-th largest, so ties at the
boundary are all kept.

1. k >= V is the unadjusted round, output for output.
2. p(x) and q(x) at the draft tokens equal a softmax over the entries that
   numpy's partition puts at or above the k-th largest (a library routine), on
   rows with heavy ties.
3. k = 1 turns sampling into greedy verify when the drafts are the draft
   argmaxes: the round then equals the oracle's greedy verify.
4. Exactness holds for the adjusted distributions: with drafts drawn from the
   adjusted q, the first emitted token follows the adjusted p (chi-square) and
   the first acceptance rate is sum_x min(p'(x), q'(x)).
5. Every emitted token lies in the target row's kept set.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import chisq_pvalue


def _kept(z, k):
    """Mask of the entries of each row at or above its k-th largest (numpy)."""
    if k >= z.shape[-1]:
        return np.ones(z.shape, bool)
    kth = -np.partition(-z, k - 1, axis=-1)[..., k - 1:k]
    return z >= kth


def _adjusted(z, k, T=1.0):
    inv_t = float(np.float32(1.0) / np.float32(T))  # the single-precision 1/T of both sides
    s = np.where(_kept(z, k), z.astype(np.float64) * inv_t, -np.inf)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _case(seed, B=8, g=3, V=40, ties=False):
    rng = np.random.default_rng(seed)
    if ties:
        zt = rng.integers(-3, 4, (B, g + 1, V)).astype(np.float32)
        zd = rng.integers(-3, 4, (B, g, V)).astype(np.float32)
    else:
        zt = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
        zd = (zt[:, :g] + rng.normal(0, 1, (B, g, V))).astype(np.float32)
    xt = rng.integers(0, V, (B, g)).astype(np.int32)
    return zt, zd, xt


@pytest.mark.parametrize("k", [40, 41, 1000])
def test_k_at_least_V_is_the_plain_round(k):
    zt, zd, xt = _case(1)
    a = oracle.spec_verify(zt, zd, xt, temperature=0.8, seed=3, rnd=1)
    b = oracle.spec_verify(zt, zd, xt, temperature=0.8, seed=3, rnd=1, top_k=k)
    for key in ("tokens", "counts", "p", "q", "ratio", "u", "flags"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


@pytest.mark.parametrize("k,ties,T", [(1, False, 1.0), (5, False, 0.7), (5, True, 1.0),
                                      (12, True, 1.3), (39, False, 1.0)])
def test_probabilities_at_drafts_match_a_library_softmax(k, ties, T):
    zt, zd, xt = _case(2 + k, ties=ties)
    out = oracle.spec_verify(zt, zd, xt, temperature=T, seed=1, rnd=0, top_k=k)
    pt = _adjusted(zt[:, :-1], k, T)
    qd = _adjusted(zd, k, T)
    B, g = xt.shape
    ref_p = np.take_along_axis(pt, xt[..., None], -1)[..., 0]
    ref_q = np.take_along_axis(qd, xt[..., None], -1)[..., 0]
    np.testing.assert_allclose(out["p"], ref_p, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(out["q"], ref_q, rtol=1e-12, atol=1e-300)


def test_k1_is_greedy_verify():
    rng = np.random.default_rng(7)
    B, g, V = 200, 4, 64
    zt = rng.normal(0, 1, (B, g + 1, V)).astype(np.float32)
    zd = (zt[:, :g] + rng.normal(0, 0.7, (B, g, V))).astype(np.float32)
    xt = zd.argmax(-1).astype(np.int32)  # the only token the adjusted q can propose
    s = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=11, rnd=4, top_k=1)
    gr = oracle.spec_verify_greedy(zt, xt)
    np.testing.assert_array_equal(s["tokens"], gr["tokens"])
    np.testing.assert_array_equal(s["counts"], gr["counts"])
    assert (s["counts"] < g).any() and (s["counts"] == g).any()


@pytest.mark.parametrize("k,seed", [(3, 21), (6, 22)])
def test_exactness_on_adjusted_distributions(k, seed):
    rng = np.random.default_rng(seed)
    V, n = 10, 200_000
    zt1 = rng.normal(0, 1.5, (1, 2, V)).astype(np.float32)
    zd1 = (zt1[:, :1] + rng.normal(0, 1.0, (1, 1, V))).astype(np.float32)
    p1 = _adjusted(zt1[0, 0], k)
    q1 = _adjusted(zd1[0, 0], k)
    zt = np.repeat(zt1, n, axis=0)
    zd = np.repeat(zd1, n, axis=0)
    xt = rng.choice(V, size=(n, 1), p=q1).astype(np.int32)
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=seed, rnd=0, top_k=k)
    first = out["tokens"][:, 0]
    obs = np.bincount(first, minlength=V)
    support = p1 > 0
    assert obs[~support].sum() == 0
    assert chisq_pvalue(obs[support], p1[support]) > 1e-3
    acc = np.minimum(p1, q1).sum()
    assert abs(np.mean(out["counts"] == 1) - acc) < 5 * np.sqrt(acc * (1 - acc) / n)


def test_emitted_tokens_are_in_the_kept_set():
    zt, zd, xt = _case(31, B=300, g=3, V=50)
    k = 4
    # drafts from the adjusted q so that most rounds test something
    rng = np.random.default_rng(5)
    qd = _adjusted(zd, k)
    xt = np.array([[rng.choice(50, p=qd[b, i]) for i in range(3)] for b in range(300)],
                  np.int32)
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=2, rnd=9, top_k=k)
    kept = _kept(zt, k)
    for b in range(300):
        n = int(out["counts"][b])
        assert kept[b, n, out["tokens"][b, n]]
        for i in range(n):
            assert out["tokens"][b, i] == xt[b, i]


def test_negative_k_rejected():
    zt, zd, xt = _case(3, B=1)
    with pytest.raises(ValueError):
        oracle.spec_verify(zt, zd, xt, top_k=-1)
