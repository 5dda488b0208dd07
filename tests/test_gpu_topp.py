"""Nucleus (top-p) adjusted verify (spec_verify_opts, top_p) on the GPU against
the oracle.

The GPU takes each row's nucleus cut with a radix select over exact fixed-point
mass sums, then runs the thresholded round; the oracle sorts each row and adds
probabilities in double.  Rules are those of tests/_parity.py, with the nucleus
near-tie rule.  Also: top_p = 1 is the plain round bit for bit, and a tiny top_p
with drafts at the draft argmax equals greedy verify.
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


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()


def both(zt, zd, xt, top_p, top_k=0, T=1.0, seed=0, rnd=0, want_alpha=False):
    g = to_np(sv.spec_verify(zt, zd, xt, temperature=T, seed=seed, round=rnd, top_p=top_p,
                             top_k=top_k, want_alpha=want_alpha))
    o = oracle.spec_verify(wl.to_oracle(zt), wl.to_oracle(zd), xt.cpu().numpy(), temperature=T,
                           seed=seed, rnd=rnd, threads=THREADS, top_p=top_p, top_k=top_k,
                           want_beta=want_alpha)
    return g, o


def case(V, B, g, dtype, seed, ties=False):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    if ties:
        zt = torch.randint(-4, 5, (B, g + 1, V), generator=gen, device="cuda").float() * 0.5
        zd = torch.randint(-4, 5, (B, g, V), generator=gen, device="cuda").float() * 0.5
    else:
        zt = torch.randn((B, g + 1, V), generator=gen, device="cuda") * 2.0
        zd = zt[:, :g] + torch.randn((B, g, V), generator=gen, device="cuda") * 0.7
    zt, zd = zt.to(dtype).contiguous(), zd.to(dtype).contiguous()
    return zt, zd, wl.draw_from_logits(zd, 1.0, gen)


@pytest.mark.parametrize("top_p,top_k", [(0.9, 0), (0.5, 0), (0.95, 200)])
def test_sample_b64_topp(top_p, top_k):
    w = wl.sample_b64(sigma=1.0)
    near = dec = 0
    for r in range(2):
        gpu, orc = both(w.zt, w.zd, w.xt, top_p, top_k, T=w.temperature, rnd=r,
                        want_alpha=(r == 0))
        n, d = assert_parity(gpu, orc, w.gamma,
                             what=f"sample_b64 top_p={top_p} top_k={top_k} round {r}")
        near, dec = near + n, dec + d
        if r == 0:
            np.testing.assert_allclose(gpu["alpha"], orc["alpha"], rtol=1e-5)
    assert near <= 1e-4 * max(dec, 1e4)


@pytest.mark.parametrize("dtype,V,top_p,ties,T", [(torch.float32, 1000, 0.8, False, 1.0),
                                                  (torch.float32, 1001, 0.6, False, 0.7),
                                                  (torch.bfloat16, 4099, 0.9, False, 1.0),
                                                  (torch.bfloat16, 2048, 0.7, True, 1.0),
                                                  (torch.float32, 3000, 0.3, True, 1.3),
                                                  (torch.bfloat16, 4099, 0.99, False, 1.0),
                                                  (torch.float32, 3000, 0.999, False, 0.7),
                                                  (torch.float32, 1000, 0.999, True, 1.0)])
def test_topp_shapes_and_ties(dtype, V, top_p, ties, T):
    B, g = 24, 3
    zt, zd, xt = case(V, B, g, dtype, seed=V, ties=ties)
    for r in range(2):
        gpu, orc = both(zt, zd, xt, top_p, T=T, seed=5, rnd=r)
        assert_parity(gpu, orc, g, what=f"top_p={top_p} V={V} {dtype} ties={ties} round {r}")


def test_top_p_one_is_the_plain_round():
    w = wl.sample_b64(sigma=1.0, B=8)
    a = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature, seed=1, round=2))
    b = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature, seed=1, round=2,
                             top_p=1.0))
    for key in ("tokens", "counts", "p", "q", "flags"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_tiny_top_p_is_greedy_verify():
    B, g, V = 64, 4, 5000
    zt, zd, _ = case(V, B, g, torch.float32, seed=9)
    xt = zd.argmax(-1).to(torch.int32).contiguous()
    s = to_np(sv.spec_verify(zt, zd, xt, temperature=1.0, seed=9, round=1, top_p=1e-6))
    gr = to_np(sv.spec_verify_greedy(zt, xt))
    np.testing.assert_array_equal(s["tokens"], gr["tokens"])
    np.testing.assert_array_equal(s["counts"], gr["counts"])
