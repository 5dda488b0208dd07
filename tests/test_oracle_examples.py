"""Pins of the oracle's accept/residual arithmetic against the pages' worked examples.

Values come from tests/golden/worked_examples.json (each entry cites its page).
The oracle works in double precision; the pages' decimals are exact in
rationals, so the tolerance is a few ulp.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import exact, theory

TOL = 1e-12


def _dist(vals):
    return np.array([float(Fraction(v)) if isinstance(v, str) else float(v) for v in vals])


def test_three_token(golden):
    g = golden("worked_examples.json")["three_token"]
    p, q = _dist(g["p"]), _dist(g["q"])
    beta, acc = oracle.accept_mass(p, q)
    np.testing.assert_allclose(acc, g["accepted_mass"], atol=TOL)
    assert abs(beta - g["accepted_total"]) < TOL
    rej, res = oracle.residual(p, q)
    assert abs(rej - g["rejection_probability"]) < TOL
    assert abs((1 - beta) - rej) < TOL  # rejection mass == residual mass
    np.testing.assert_allclose(res, g["residual_normalised"], atol=TOL)
    np.testing.assert_allclose(acc + rej * res, g["final_distribution"], atol=TOL)


def test_three_token_equal_and_disjoint(golden):
    ge = golden("worked_examples.json")["three_token_equal"]
    p, q = _dist(ge["p"]), _dist(ge["q"])
    rej, res = oracle.residual(p, q)
    assert rej == ge["rejection_probability"]
    assert np.all(res == 0)  # zero-mass residual left unnormalised
    gd = golden("worked_examples.json")["disjoint"]
    p, q = _dist(gd["p"]), _dist(gd["q"])
    beta, acc = oracle.accept_mass(p, q)
    rej, res = oracle.residual(p, q)
    assert rej == gd["rejection_probability"] and beta == 0.0
    np.testing.assert_allclose(acc + rej * res, gd["final_distribution"], atol=TOL)


def test_four_token(golden):
    g = golden("worked_examples.json")["four_token"]
    p, q = np.array(g["p"]), np.array(g["q"])
    beta, acc = oracle.accept_mass(p, q)
    assert abs(beta - g["beta"]) < TOL
    rej, res = oracle.residual(p, q)
    assert abs(rej - g["rejection_probability"]) < TOL
    np.testing.assert_allclose(np.maximum(p - q, 0), g["residual_unnormalised"], atol=TOL)
    np.testing.assert_allclose(res, g["residual_normalised"], atol=TOL)
    assert abs(rej * res[0] - g["token0_via_rejection"]) < TOL
    total = acc + rej * res
    assert abs(total[0] - g["token0_total"]) < TOL
    assert abs(total[1] - g["token1_total"]) < TOL
    assert abs(min(1.0, p[1] / q[1]) - g["accept_prob_token1"]) < TOL
    # Appendix A.2 comparison: 1/r_max = 0.60 is below beta = 0.75
    r = theory.rejection_sampling_rate(p, q)
    assert abs(r - g["rejection_sampling_rate"]) < TOL and r < beta


def test_cat_dog_owl(golden):
    g = golden("worked_examples.json")["cat_dog_owl"]
    p, q = np.array(g["p"]), np.array(g["q"])
    beta, acc = oracle.accept_mass(p, q)
    np.testing.assert_allclose(acc, g["kept"], atol=TOL)
    assert abs(beta - g["kept_total"]) < TOL
    rej, res = oracle.residual(p, q)
    np.testing.assert_allclose(rej * res, g["repair"], atol=TOL)
    np.testing.assert_allclose(acc + rej * res, g["final_distribution"], atol=TOL)


@pytest.mark.parametrize("seed", range(20))
def test_accept_plus_residual_is_p_random(seed):
    """min(p,q) + (1-beta) p' == p for random p, q (course notes, 'Exactness')."""
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 40))
    p = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 2))
    q = rng.dirichlet(np.ones(V) * rng.uniform(0.1, 2))
    if seed % 3 == 0:
        q[rng.integers(0, V, size=V // 3)] = 0
        q /= q.sum()
    beta, acc = oracle.accept_mass(p, q)
    rej, res = oracle.residual(p, q)
    assert abs(beta + rej - 1) < 1e-12
    np.testing.assert_allclose(acc + rej * res, p, atol=1e-12)
    # alpha = 1 - TV (course notes, 'How often do we accept?')
    assert abs(beta - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12


def test_exact_rational_round_trip(golden):
    """The exact-enumeration helper's residual agrees with the three-token page in rationals."""
    g = golden("worked_examples.json")["three_token"]
    p = [Fraction(v) for v in g["p"]]
    q = [Fraction(v) for v in g["q"]]
    res = exact.residual(p, q)
    assert res == [Fraction(1), Fraction(0), Fraction(0)]
    assert exact.residual(p, p) is None


def test_softmax_closed_forms():
    # constant logits -> uniform; logits = log p -> p
    S, pr = oracle.softmax(np.zeros(7))
    assert S == 7.0 and np.allclose(pr, 1 / 7, atol=1e-15)
    p = np.array([0.5, 0.25, 0.125, 0.125])
    S, pr = oracle.softmax(np.log(p))
    np.testing.assert_allclose(pr, p, atol=1e-15)
    S, pr = oracle.softmax(np.array([-np.inf, -np.inf]))
    assert S == 0.0 and np.all(pr == 0)
