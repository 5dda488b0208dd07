"""Statistical pins of the oracle's full verify (logits in, tokens out).

The oracle is run as a sampler with its own Philox streams; draft tokens are
drawn from q with numpy's RNG (an independent generator).  What the pages fix:
  * the emitted token is distributed as p (course notes, 'Exactness'; the
    three-token example of the lihaoran.work essay, p = (0.6, 0.3, 0.1));
  * the acceptance rate is sum min(p,q) = 1 - TV (course notes, 'How often do
    we accept?');
  * with identical (p, q) at every position the number of tokens per round
    follows equation (1) and the Figure 4 histogram ('Fast Inference ...',
    'Tokens per target run, equation (1)'): 3.60 tokens at alpha=0.75, gamma=7.
"""
import numpy as np
import pytest

import oracle
from oracle import theory
from tests._helpers import chisq_pvalue, logits_from_probs, sample_rows

P3 = [0.6, 0.3, 0.1]
Q3 = [0.2, 0.5, 0.3]


def _single_position_run(p, q, n, seed, rnd=0, dtype="f32"):
    rng = np.random.default_rng(seed)
    V = len(p)
    zt = np.empty((n, 2, V), np.float32)
    zt[:, 0] = logits_from_probs(p)
    zt[:, 1] = logits_from_probs(p)
    zd = np.empty((n, 1, V), np.float32)
    zd[:, 0] = logits_from_probs(q)
    xt = sample_rows(rng, np.broadcast_to(np.asarray(q, float), (n, 1, V)))
    return oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=seed, rnd=rnd), xt


def test_three_token_chi_square_1e6():
    out, xt = _single_position_run(P3, Q3, 1_000_000, seed=11)
    first = out["tokens"][:, 0]
    counts = np.bincount(first, minlength=3)
    assert chisq_pvalue(counts, P3) > 1e-3
    # acceptance frequency = 1 - TV = 0.6, within 4 sigma
    acc = (out["counts"] == 1).mean()
    assert abs(acc - 0.6) < 4 * np.sqrt(0.6 * 0.4 / 1e6)
    # every rejection is corrected to token 0 (all residual mass on it)
    rej = out["counts"] == 0
    assert np.all(out["tokens"][rej, 0] == 0)
    # p(x~), q(x~) are exact softmax values of the logits
    np.testing.assert_allclose(out["p"][:, 0], np.asarray(P3)[xt[:, 0]], rtol=1e-6)
    np.testing.assert_allclose(out["q"][:, 0], np.asarray(Q3)[xt[:, 0]], rtol=1e-6)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_v8_with_draft_zeros(seed):
    rng = np.random.default_rng(100 + seed)
    V = 8
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.7)
    q[rng.choice(V, 2, replace=False)] = 0.0  # tokens the draft never proposes
    q /= q.sum()
    n = 400_000
    out, _ = _single_position_run(p, q, n, seed=seed)
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert chisq_pvalue(counts, p) > 1e-3
    alpha = np.minimum(p, q).sum()
    acc = (out["counts"] == 1).mean()
    assert abs(acc - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / n)
    assert abs(alpha - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12


def test_equation1_and_histogram_four_token():
    p = [0.50, 0.30, 0.15, 0.05]  # 'Fast Inference ...', four-token example: beta = 0.75
    q = [0.30, 0.50, 0.10, 0.10]
    gamma, n, V = 7, 100_000, 4
    rng = np.random.default_rng(7)
    zt = np.broadcast_to(logits_from_probs(p), (n, gamma + 1, V)).copy()
    zd = np.broadcast_to(logits_from_probs(q), (n, gamma, V)).copy()
    xt = sample_rows(rng, np.broadcast_to(np.asarray(q), (n, gamma, V)))
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=3, rnd=5)
    tokens = out["counts"] + 1
    mean = tokens.mean()
    expect = theory.expected_tokens(0.75, gamma)
    assert abs(expect - 3.60) < 0.005  # the page's number
    assert abs(mean - expect) < 4 * tokens.std() / np.sqrt(n)
    hist = np.bincount(tokens, minlength=gamma + 2)[1:]
    assert chisq_pvalue(hist, theory.tokens_histogram(0.75, gamma)) > 1e-3
    # structure of the output rows
    for b in range(200):
        k = out["counts"][b]
        assert np.array_equal(out["tokens"][b, :k], xt[b, :k])
        assert np.all(out["tokens"][b, k + 1:] == -1)
        assert 0 <= out["tokens"][b, k] < V


def test_temperature_rescales_both_rows():
    """At T=2 the oracle verifies against softmax(z/2) for target and draft alike."""
    rng = np.random.default_rng(5)
    V, n = 6, 300_000
    zt_row = rng.normal(0, 2, V).astype(np.float32)
    zd_row = rng.normal(0, 2, V).astype(np.float32)
    T = 2.0
    inv = np.float64(np.float32(1.0) / np.float32(T))
    p = np.exp(zt_row * inv - (zt_row * inv).max()); p /= p.sum()
    q = np.exp(zd_row * inv - (zd_row * inv).max()); q /= q.sum()
    zt = np.broadcast_to(np.stack([zt_row, zt_row]), (n, 2, V)).copy()
    zd = np.broadcast_to(zd_row, (n, 1, V)).copy()
    xt = sample_rows(rng, np.broadcast_to(q, (n, 1, V)))
    out = oracle.spec_verify(zt, zd, xt, temperature=T, seed=9)
    assert chisq_pvalue(np.bincount(out["tokens"][:, 0], minlength=V), p) > 1e-3
    np.testing.assert_allclose(out["p"][:, 0], p[xt[:, 0]], rtol=1e-12)
    # per-row temperature gives the same result as the scalar
    out2 = oracle.spec_verify(zt[:1000], zd[:1000], xt[:1000], temperature=9.0,
                              row_temperature=np.full(1000, T, np.float32), seed=9)
    np.testing.assert_array_equal(out2["tokens"], out["tokens"][:1000])


def test_beta_diagnostic_is_overlap():
    rng = np.random.default_rng(8)
    V, g = 16, 3
    zt = rng.normal(0, 1.5, (4, g + 1, V)).astype(np.float32)
    zd = (zt[:, :g] + rng.normal(0, 1, (4, g, V))).astype(np.float32)
    xt = rng.integers(0, V, (4, g)).astype(np.int32)
    out = oracle.spec_verify(zt, zd, xt, temperature=1.0, seed=1, want_beta=True)
    for b in range(4):
        for i in range(g):
            _, p = oracle.softmax(zt[b, i].astype(np.float64))
            _, q = oracle.softmax(zd[b, i].astype(np.float64))
            assert abs(out["beta"][b, i] - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
        n = out["counts"][b]
        if n < g:  # 1 - (residual mass) equals beta at the rejected position
            assert abs(out["resid_mass"][b] - (1 - out["beta"][b, n])) < 1e-12
    np.testing.assert_allclose(out["alpha"], out["beta"].mean(axis=1))
