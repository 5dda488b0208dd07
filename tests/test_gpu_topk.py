"""Top-k adjusted verify (spec_verify_opts, top_k) on the GPU against the oracle.

The GPU finds each row's threshold from candidates at or above the k-th largest
chunk max (or, for large k, many candidates or ties, by radix passes over the
row) and masks the tail in the decision, the draw and the overlap; the oracle
sorts each row.
Rules are those of tests/_parity.py.  Also: k >= V is the plain round bit for
bit, and k = 1 with drafts at the draft argmax equals greedy verify.
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


def both(zt, zd, xt, k, T=1.0, seed=0, rnd=0, want_alpha=False):
    g = to_np(sv.spec_verify(zt, zd, xt, temperature=T, seed=seed, round=rnd, top_k=k,
                             want_alpha=want_alpha))
    o = oracle.spec_verify(wl.to_oracle(zt), wl.to_oracle(zd), xt.cpu().numpy(), temperature=T,
                           seed=seed, rnd=rnd, threads=THREADS, top_k=k, want_beta=want_alpha)
    return g, o


def kept_draws(zd, k, gen):
    """Draft tokens drawn from the top-k adjusted draft rows."""
    kth = torch.topk(zd.float(), k, dim=-1).values[..., -1:]
    z = torch.where(zd.float() >= kth, zd.float(), torch.full_like(zd.float(), float("-inf")))
    return wl.draw_from_logits(z, 1.0, gen)


def case(V, B, g, dtype, seed, ties=False):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    if ties:
        zt = torch.randint(-4, 5, (B, g + 1, V), generator=gen, device="cuda").float() * 0.5
        zd = torch.randint(-4, 5, (B, g, V), generator=gen, device="cuda").float() * 0.5
    else:
        zt = torch.randn((B, g + 1, V), generator=gen, device="cuda") * 2.0
        zd = zt[:, :g] + torch.randn((B, g, V), generator=gen, device="cuda") * 0.7
    return zt.to(dtype).contiguous(), zd.to(dtype).contiguous(), gen


@pytest.mark.parametrize("k", [1, 50, 1000])
def test_sample_b64_topk(k):
    w = wl.sample_b64(sigma=1.0)
    gen = torch.Generator(device="cuda").manual_seed(77)
    xt = kept_draws(w.zd, k, gen)
    near = dec = 0
    for r in range(2):
        gpu, orc = both(w.zt, w.zd, xt, k, T=w.temperature, rnd=r, want_alpha=(r == 0))
        n, d = assert_parity(gpu, orc, w.gamma, what=f"sample_b64 top_k={k} round {r}")
        near, dec = near + n, dec + d
        if r == 0:
            np.testing.assert_allclose(gpu["alpha"], orc["alpha"], rtol=1e-5)
    assert near <= 1e-4 * max(dec, 1e4)


@pytest.mark.parametrize("dtype,V,k,ties", [(torch.float32, 1000, 7, False),
                                            (torch.float32, 1001, 7, False),
                                            (torch.bfloat16, 4099, 33, False),
                                            (torch.bfloat16, 2048, 10, True),
                                            (torch.float32, 3000, 100, True),
                                            (torch.float32, 64, 63, False),
                                            (torch.bfloat16, 40000, 10, False),
                                            (torch.bfloat16, 40000, 10, True),
                                            (torch.float32, 30000, 5, False)])
def test_topk_shapes_and_ties(dtype, V, k, ties):
    B, g = 24, 3
    zt, zd, gen = case(V, B, g, dtype, seed=V + k, ties=ties)
    xt = kept_draws(zd, k, gen)
    for r in range(2):
        gpu, orc = both(zt, zd, xt, k, T=0.9, seed=3, rnd=r)
        assert_parity(gpu, orc, g, what=f"top_k={k} V={V} {dtype} ties={ties} round {r}")


@pytest.mark.parametrize("k", [128256, 200000])
def test_k_at_least_V_is_the_plain_round(k):
    w = wl.sample_b64(sigma=1.0, B=8)
    a = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature, seed=1, round=2))
    b = to_np(sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature, seed=1, round=2,
                             top_k=k))
    for key in ("tokens", "counts", "p", "q", "flags"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_k1_is_greedy_verify():
    B, g, V = 64, 4, 5000
    zt, zd, _ = case(V, B, g, torch.float32, seed=5)
    xt = zd.argmax(-1).to(torch.int32).contiguous()
    s = to_np(sv.spec_verify(zt, zd, xt, temperature=1.0, seed=9, round=1, top_k=1))
    gr = to_np(sv.spec_verify_greedy(zt, xt))
    np.testing.assert_array_equal(s["tokens"], gr["tokens"])
    np.testing.assert_array_equal(s["counts"], gr["counts"])
    assert (s["counts"] < g).any()
