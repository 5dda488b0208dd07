"""The target's own draw by the inverse transform, pinned.

"Fast Inference from Transformers via Speculative Decoding", section "The loop",
step 3: after a rejection at n the target samples one token from the residual
norm(max(0, p_n - q_n)), after a clean sweep from p_{gamma+1}; the pages leave
the sampling method open.  The oracle draws U in [0, 1) with 53 random bits
(Philox tag 1 at the draw position) and takes the smallest v, in vocabulary
order, whose cumulative weight exceeds U times the total.

1. Residual and bonus draws on random rows equal numpy's searchsorted over
   numpy's cumulative sums of the same distribution (scipy softmax), with U
   read back from the oracle.
2. The pages' four-token example: residual (0.8, 0, 0.2, 0) gives token 0 for
   U < 0.8 and token 2 otherwise.
3. U is uniform on [0, 1) (Kolmogorov-Smirnov over many batch rows) and
   depends on the counter words it names: position, batch row and round.
4. The reported gap is the distance of U W to the nearer end of the drawn
   token's interval.
"""
import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle


def _round(zt, zd, xt, seed, rnd, T=1.0):
    return oracle.spec_verify(zt.astype(np.float32), zd.astype(np.float32), xt.astype(np.int32),
                              temperature=T, seed=seed, rnd=rnd, sampler="inverse")


def _searchsorted_draw(w, U):
    C = np.cumsum(w)
    t = U * C[-1]
    v = int(np.searchsorted(C, t, side="right"))
    lo = C[v - 1] if v > 0 else 0.0
    return v, min(t - lo, C[v] - t)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_residual_draw_is_searchsorted(seed):
    """gamma = 1 and a draft token with p(x) = 0: every batch row rejects at 0
    and draws from max(0, p_0 - q_0)."""
    rng = np.random.default_rng(seed)
    B, V, T = 300, 97, 0.8
    zt = rng.normal(0, 1.5, (B, 2, V))
    zd = (zt[:, :1] + rng.normal(0, 1.0, (B, 1, V)))
    xt = rng.integers(0, V, (B, 1))
    zt[np.arange(B), 0, xt[:, 0]] = -np.inf
    out = _round(zt, zd, xt, seed, rnd=5, T=T)
    assert np.all(out["counts"] == 0)
    invT = float(np.float32(1.0) / np.float32(T))
    checked = 0
    for b in range(B):
        p = softmax(zt[b, 0].astype(np.float32).astype(np.float64) * invT)
        q = softmax(zd[b, 0].astype(np.float32).astype(np.float64) * invT)
        w = np.maximum(p - q, 0.0)
        U = oracle.draw_uniform(seed, 0, b, 5)
        v, gap = _searchsorted_draw(w, U)
        if gap < 1e-12:
            continue
        assert out["tokens"][b, 0] == v, (b, U)
        np.testing.assert_allclose(out["gap"][b], gap, rtol=1e-9, atol=1e-15)
        checked += 1
    assert checked > B - 3


@pytest.mark.parametrize("seed", [4, 5])
def test_bonus_draw_is_searchsorted(seed):
    """Draft row equal to target row 0 and x at a positive-probability entry: the
    ratio is 1, the draft is accepted, and the bonus token comes from p_1."""
    rng = np.random.default_rng(seed)
    B, V = 300, 64
    zt = rng.normal(0, 2.0, (B, 2, V)).astype(np.float32)
    zd = zt[:, :1].copy()
    xt = rng.integers(0, V, (B, 1))
    out = _round(zt, zd, xt, seed, rnd=2)
    assert np.all(out["counts"] == 1)
    for b in range(B):
        p1 = softmax(zt[b, 1].astype(np.float64))
        v, gap = _searchsorted_draw(p1, oracle.draw_uniform(seed, 1, b, 2))
        if gap < 1e-12:
            continue
        assert out["tokens"][b, 1] == v
        assert out["tokens"][b, 0] == xt[b, 0]


def test_four_token_worked_example():
    """p = (0.5, 0.3, 0.15, 0.05), q = (0.3, 0.5, 0.1, 0.1): the residual is
    (0.8, 0, 0.2, 0) once normalised (the four-token example of the accept/reject
    section), so the draw is token 0 iff U < 0.8.  The draft token 1 has
    p/q = 0.6; rows whose acceptance uniform exceeds 0.6 reject."""
    p = np.array([0.5, 0.3, 0.15, 0.05])
    q = np.array([0.3, 0.5, 0.1, 0.1])
    B = 400
    zt = np.tile(np.log(p), (B, 2, 1))
    zd = np.tile(np.log(q), (B, 1, 1))
    xt = np.ones((B, 1))
    out = _round(zt, zd, xt, seed=8, rnd=1)
    rejected = out["counts"] == 0
    assert 0.3 < rejected.mean() < 0.5  # 1 - 0.6
    seen = set()
    for b in np.nonzero(rejected)[0]:
        U = oracle.draw_uniform(8, 0, int(b), 1)
        if abs(U - 0.8) < 1e-9:
            continue
        want = 0 if U < 0.8 else 2
        assert out["tokens"][b, 0] == want
        seen.add(want)
    assert seen == {0, 2}


def test_draw_uniform_is_uniform_and_keyed():
    us = np.array([oracle.draw_uniform(11, 0, b, 0) for b in range(20000)])
    assert np.all((us >= 0.0) & (us < 1.0))
    assert stats.kstest(us, "uniform").pvalue > 1e-3
    base = oracle.draw_uniform(11, 2, 7, 3)
    for other in (oracle.draw_uniform(12, 2, 7, 3), oracle.draw_uniform(11, 3, 7, 3),
                  oracle.draw_uniform(11, 2, 8, 3), oracle.draw_uniform(11, 2, 7, 4)):
        assert other != base


def test_draw_uniform_counter_words():
    """U = k 2^-53 with k from words 0 and 1 of Philox4x32-10 at counter
    (0, 1<<24 | pos, b, round) under key (lo32 seed, hi32 seed)."""
    seed, pos, b, rnd = 0x1234_5678_9ABC_DEF0, 3, 41, 77
    w = oracle.philox4x32_10([0, (1 << 24) | pos, b, rnd], [seed & 0xFFFFFFFF, seed >> 32])
    k = (int(w[0]) >> 11 << 32) | int(w[1])
    assert oracle.draw_uniform(seed, pos, b, rnd) == k / 2.0**53
