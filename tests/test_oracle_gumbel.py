"""The target's own draw by Gumbel-max (the oracle's default sampler), pinned.

"Fast Inference from Transformers via Speculative Decoding", section "The loop",
step 3: after a rejection at n the target samples one token from the residual
norm(max(0, p_n - q_n)), after a clean sweep from p_{gamma+1}.  The oracle takes
the argmax over the entries of positive weight of log w_v + g_v, with g_v =
-log(-log u_v) and u_v from Philox tag 1 at the draw position (counter word 0 =
v>>2, lane v&3), ties to the lowest index.

What fixes it (none of these retypes the oracle's formula):
1. The residual draw is distributed as norm(max(0, p - q)) and the bonus draw as
   p (chi-square against scipy softmax rows, one independent noise stream per
   batch row).
2. The four-token example of the accept/reject section: the residual
   (0.8, 0, 0.2, 0) puts tokens on 0 and 2 only, in that ratio.
3. The reported margin (top-1 minus top-2 key) is exponential with mean 1 on
   wide rows of equal weights: the spacing of the two largest of many i.i.d.
   standard Gumbel variables (a planted noise of the wrong law, or a key without
   the log of the weight, fails it).
4. The noise depends on the counter words the contract names (position, batch
   row, round, seed) and not on the draft side's tag.
A last test checks the counter layout itself against the pinned Philox uniforms
(a contract check, not a pin).
"""
import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle
from tests._helpers import chisq_pvalue


def _round(zt, zd, xt, seed, rnd, T=1.0):
    return oracle.spec_verify(zt.astype(np.float32), zd.astype(np.float32), xt.astype(np.int32),
                              temperature=T, seed=seed, rnd=rnd)


def _always_reject(p, q, B):
    """gamma = 1 rows whose draft token has p = 0: every row rejects at 0 and
    draws from max(0, p - q) (the draft token carries q mass, so q keeps it)."""
    V = len(p)
    x = int(np.argmax(q))
    pt = np.asarray(p, float).copy()
    pt[x] = 0.0
    pt /= pt.sum()
    with np.errstate(divide="ignore"):
        zt = np.tile(np.log(pt), (B, 2, 1))
        zd = np.tile(np.log(np.asarray(q, float)), (B, 1, 1))
    xt = np.full((B, 1), x)
    return zt, zd, xt, pt


@pytest.mark.parametrize("seed", [1, 2])
def test_residual_draw_distribution(seed):
    rng = np.random.default_rng(seed)
    V, B = 12, 200_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.5)
    zt, zd, xt, pt = _always_reject(p, q, B)
    out = _round(zt, zd, xt, seed, rnd=3)
    assert np.all(out["counts"] == 0)
    # the residual of the rows as the oracle reads them (float32 logits)
    pr = softmax(zt[0, 0].astype(np.float32).astype(np.float64))
    qr = softmax(zd[0, 0].astype(np.float32).astype(np.float64))
    r = np.maximum(pr - qr, 0.0)
    r /= r.sum()
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    assert np.all(counts[r == 0] == 0)
    assert chisq_pvalue(counts, r) > 1e-3


def test_bonus_draw_distribution():
    rng = np.random.default_rng(4)
    V, B = 10, 200_000
    z = rng.normal(0, 1.5, V)
    zt = np.tile(z, (B, 2, 1))
    zd = zt[:, :1].copy()
    xt = np.full((B, 1), int(np.argmax(z)))  # ratio 1: always accepted
    out = _round(zt, zd, xt, 5, rnd=0, T=0.7)
    assert np.all(out["counts"] == 1)
    invT = float(np.float32(1.0) / np.float32(0.7))
    p = softmax(z.astype(np.float32).astype(np.float64) * invT)
    assert chisq_pvalue(np.bincount(out["tokens"][:, 1], minlength=V), p) > 1e-3


def test_four_token_worked_example():
    """p = (0.5, 0.3, 0.15, 0.05), q = (0.3, 0.5, 0.1, 0.1) (the four-token example
    of the accept/reject section): draft token 1 has p/q = 0.6; after a rejection
    the residual normalises to (0.8, 0, 0.2, 0)."""
    p = np.array([0.5, 0.3, 0.15, 0.05])
    q = np.array([0.3, 0.5, 0.1, 0.1])
    B = 100_000
    zt = np.tile(np.log(p), (B, 2, 1))
    zd = np.tile(np.log(q), (B, 1, 1))
    xt = np.ones((B, 1))
    out = _round(zt, zd, xt, seed=8, rnd=1)
    rej = out["counts"] == 0
    n = int(rej.sum())
    assert abs(n / B - 0.4) < 4 * np.sqrt(0.24 / B)
    t = out["tokens"][rej, 0]
    assert set(np.unique(t).tolist()) == {0, 2}
    counts = np.bincount(t, minlength=4)
    assert chisq_pvalue(counts[[0, 2]], [0.8, 0.2]) > 1e-3


def test_margin_is_standard_exponential():
    """Equal weights over V entries: the keys are i.i.d. standard Gumbel plus a
    constant, and the top-1 minus top-2 spacing is exponential with mean 1 (up
    to a factor V/(V-1) in its rate)."""
    B, V = 6000, 2048
    zt = np.zeros((B, 2, V))
    zd = np.zeros((B, 1, V))
    xt = np.zeros((B, 1))
    out = _round(zt, zd, xt, seed=21, rnd=4)
    assert np.all(out["counts"] == 1)  # p = q: accepted, then the bonus draw
    gap = out["gap"]
    # 23-bit uniforms: two entries of a row may draw the same u (a tie, margin 0,
    # decided for the lower index), about once per 4096 rows at this width
    assert np.all(gap >= 0) and np.mean(gap == 0) < 2e-3
    assert stats.kstest(gap, "expon").pvalue > 1e-3
    # the drawn token is uniform over the row
    assert chisq_pvalue(np.bincount(out["tokens"][:, 1] // 64, minlength=V // 64),
                        np.full(V // 64, 64 / V)) > 1e-3


def test_noise_is_keyed_by_the_counter():
    B, V = 64, 4096
    zt = np.zeros((B, 2, V))
    zd = np.zeros((B, 1, V))
    xt = np.zeros((B, 1))
    base = _round(zt, zd, xt, seed=3, rnd=9)["tokens"][:, 1]
    assert len(set(base.tolist())) > B // 2          # batch rows draw apart
    for kw in (dict(seed=4, rnd=9), dict(seed=3, rnd=10)):
        other = _round(zt, zd, xt, **kw)["tokens"][:, 1]
        assert np.mean(other == base) < 0.1
    # position: gamma = 2 with both drafts accepted draws at position 2
    zt3 = np.zeros((B, 3, V))
    zd3 = np.zeros((B, 2, V))
    t3 = _round(zt3, zd3, np.zeros((B, 2)), seed=3, rnd=9)["tokens"][:, 2]
    assert np.mean(t3 == base) < 0.1
    # the draft side's tag-2 stream is a different stream
    d = oracle.draft_sample(np.zeros((B, V), np.float32), seed=3, rnd=9, pos=1)["tokens"]
    assert np.mean(d == base) < 0.1


def test_counter_layout_contract():
    """The drawn token is the argmax of log w_v - log(-log u_v) with u_v the pinned
    Philox uniform at (tag 1, the draw position, b, round; word v>>2, lane v&3)."""
    rng = np.random.default_rng(12)
    B, V, seed, rnd = 40, 37, 77, 6
    zt = rng.normal(0, 1.0, (B, 2, V))
    zd = zt[:, :1] + rng.normal(0, 1.0, (B, 1, V))
    xt = rng.integers(0, V, (B, 1))
    out = _round(zt, zd, xt, seed, rnd)
    for b in range(B):
        n = int(out["counts"][b])
        p = softmax(zt[b, n].astype(np.float32).astype(np.float64))
        if n == 0:
            q = softmax(zd[b, 0].astype(np.float32).astype(np.float64))
            w = np.maximum(p - q, 0.0)
        else:
            w = p
        u = oracle.uniform_row(seed, 1, n, b, rnd, 0, V)
        with np.errstate(divide="ignore"):
            key = np.where(w > 0, np.log(w) - np.log(-np.log(u)), -np.inf)
        top = np.sort(key)[::-1]
        if top[0] - top[1] < 1e-9:
            continue
        assert out["tokens"][b, n] == int(np.argmax(key))
        np.testing.assert_allclose(out["gap"][b], top[0] - top[1], rtol=1e-7, atol=1e-12)
