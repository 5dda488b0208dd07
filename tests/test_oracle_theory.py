"""Pins for the closed forms the oracle's statistical tests rely on.

Every expected number is one the pages print (tests/golden/closed_forms.json).
"""
import pytest

from oracle import theory


def test_expected_tokens(golden):
    g = golden("closed_forms.json")["expected_tokens"]
    for a, gam, val in g["cases"]:
        assert abs(theory.expected_tokens(a, gam) - val) <= g["abs_tol"]


def test_expected_tokens_cap(golden):
    g = golden("closed_forms.json")["expected_tokens_cap"]
    for a, cap in g["cases"]:
        assert abs(theory.expected_tokens(a, 10_000) - cap) <= g["abs_tol"]
        # the cap is approached from below for every finite gamma
        assert theory.expected_tokens(a, 50) < cap


def test_tokens_histogram(golden):
    g = golden("closed_forms.json")["tokens_histogram"]
    h = theory.tokens_histogram(g["alpha"], g["gamma"])
    assert len(h) == g["gamma"] + 1
    assert abs(sum(h) - 1.0) < 1e-12
    assert abs(h[-1] - g["p_all"]) <= g["abs_tol"]
    assert abs(h[0] - g["p_one"]) <= g["abs_tol"]
    # the histogram's mean is equation (1)
    mean = sum((k + 1) * hk for k, hk in enumerate(h))
    assert abs(mean - theory.expected_tokens(g["alpha"], g["gamma"])) < 1e-12


def test_speedup_example(golden):
    g = golden("closed_forms.json")["speedup"]
    assert abs(theory.expected_tokens(g["alpha"], g["gamma"]) - g["numerator"]) <= g["abs_tol"]
    assert abs(g["gamma"] * g["c"] + 1 - g["denominator"]) <= g["abs_tol"]
    assert abs(theory.speedup(g["alpha"], g["gamma"], g["c"]) - g["value"]) <= g["abs_tol"]


def test_t5_large(golden):
    g = golden("closed_forms.json")["t5_large"]
    assert abs(theory.expected_tokens(g["alpha"], g["gamma"]) - g["numerator"]) <= g["abs_tol"]
    assert abs(g["gamma"] * g["c"] + 1 - g["denominator"]) <= g["abs_tol"]


def test_bigram(golden):
    g = golden("closed_forms.json")["bigram"]
    assert abs(theory.speedup(g["alpha"], g["gamma"], g["c"]) - g["value"]) <= g["abs_tol"]


def test_table1(golden):
    g = golden("closed_forms.json")["table1"]
    for a, gam, speed, ops in g["rows"]:
        assert abs(theory.speedup(a, gam, 0.0) - speed) <= g["abs_tol"]
        assert abs(theory.ops_factor(a, gam, 0.0) - ops) <= g["abs_tol"]


def test_corollary_gamma1(golden):
    for a, c in golden("closed_forms.json")["corollary_gamma1"]["cases"]:
        assert theory.speedup(a, 1, c) == pytest.approx((1 + a) / (1 + c), rel=1e-12)
        assert (theory.speedup(a, 1, c) > 1.0) == (a > c)
