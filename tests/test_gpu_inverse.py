"""The opt-in inverse-transform sampler (sv_options.sampler = SV_SAMPLER_INVERSE)
against the oracle's inverse transform (GPU).

The token is the smallest v whose cumulative weight exceeds U times the total,
U from one 53-bit Philox uniform.  The GPU forms fp32 weights (about 3e-7
relative error each from exp2 and the scaled logit), adds runs of at most 16 of
them in fp32 (at most 15 roundings of 2^-24 relative) and the runs exactly in
fixed point, so an interval end moves by at most about 1e-6 of the total: a
draw may differ from the oracle's only where U W lies within 4e-6 (probability
units) of an end of the drawn token's interval.  That window belongs to this
sampler alone; the default Gumbel-max draw keeps the 1e-6 key-gap rule.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_21_gb300 as sv
from speculative_decoding_verification_21_gb300 import workloads as wl
from tests._parity import assert_parity, to_np

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))
INVERSE_NEAR_DRAW = 4e-6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()


def both(w, seed, rnd, top_k=0):
    g = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature,
                             row_temperature=w.row_temperature, seed=seed, round=rnd,
                             top_k=top_k, sampler="inverse"))
    rowT = None if w.row_temperature is None else w.row_temperature.cpu().numpy()
    o = oracle.spec_verify(wl.to_oracle(w.zt), wl.to_oracle(w.zd), w.xt.cpu().numpy(),
                           temperature=w.temperature, row_temperature=rowT, seed=seed, rnd=rnd,
                           threads=THREADS, top_k=top_k, sampler="inverse")
    return g, o


@pytest.mark.parametrize("sigma", [0.25, 4.0])
def test_inverse_sample_b64(sigma):
    w = wl.sample_b64(sigma=sigma)
    for r in range(3):
        g, o = both(w, 0, r)
        assert_parity(g, o, w.gamma, what=f"inverse sigma={sigma} round {r}",
                      near_draw=INVERSE_NEAR_DRAW)


def test_inverse_ragged_and_topk():
    w = wl.sample_b64(sigma=1.0, B=8, gamma=3, V=20011)
    for r in range(3):
        g, o = both(w, 5, r)
        assert_parity(g, o, w.gamma, what=f"inverse V=20011 round {r}",
                      near_draw=INVERSE_NEAR_DRAW)
        g, o = both(w, 5, r, top_k=40)
        assert_parity(g, o, w.gamma, what=f"inverse top-k round {r}",
                      near_draw=INVERSE_NEAR_DRAW)


def test_inverse_and_gumbel_differ():
    """The two samplers are different streams: same decisions, different tokens."""
    w = wl.sample_b64(sigma=4.0)
    a = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature, seed=0, round=0))
    b = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature, seed=0, round=0,
                             sampler="inverse"))
    np.testing.assert_array_equal(a["counts"], b["counts"])
    np.testing.assert_array_equal(a["p"], b["p"])
    rows = np.arange(w.B)
    drawn_a = a["tokens"][rows, a["counts"]]
    drawn_b = b["tokens"][rows, b["counts"]]
    assert np.mean(drawn_a == drawn_b) < 0.5
