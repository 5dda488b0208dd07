"""Draft LM head + draw of a draft position (spec_lmhead_draft) on the GPU.

The logits the kernel used (debug_logits) are within 2e-2 absolute of an fp32
reference of h W; the drawn tokens are compared with the oracle's draw on those
identical logits (bit for bit except near-ties of the Gumbel keys, gap < 1e-6),
and q(x), lse within 1e-5.  A call without debug_logits gives the same result.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_21_gb300 as sv
from speculative_decoding_verification_21_gb300 import workloads as wl
from tests._helpers import chisq_pvalue

pytestmark = pytest.mark.gpu
LOGIT_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.backends.cuda.matmul.allow_tf32 = False
    sv.load()


def make(B, Hd, V, seed, wstd=0.02):
    g = torch.Generator(device="cuda").manual_seed(seed)
    h = torch.randn((B, Hd), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((Hd, V), generator=g, device="cuda") * wstd).to(torch.bfloat16)
    return h, W


def check(h, W, T, seed, rnd, pos):
    B, V = h.shape[0], W.shape[1]
    dbg = torch.full((B, V), float("nan"), device="cuda")
    o = sv.spec_lmhead_draft(h, W, pos=pos, temperature=T, seed=seed, round=rnd,
                             debug_logits=dbg)
    torch.cuda.synchronize()
    assert torch.isfinite(dbg).all()
    ref = h.float() @ W.float()
    assert (dbg - ref).abs().max().item() <= LOGIT_TOL
    orc = oracle.draft_sample(dbg.cpu().numpy(), temperature=T, seed=seed, rnd=rnd, pos=pos)
    tok = o["tokens"].cpu().numpy()
    diff = tok != orc["tokens"]
    assert np.all(orc["gap"][diff] < 1e-6), (np.nonzero(diff), orc["gap"][diff])
    same = ~diff
    np.testing.assert_allclose(o["q"].cpu().numpy()[same], orc["q"][same], rtol=1e-5, atol=1e-30)
    np.testing.assert_allclose(o["lse"].cpu().numpy(), orc["lse"], rtol=1e-5, atol=1e-5)
    o2 = sv.spec_lmhead_draft(h, W, pos=pos, temperature=T, seed=seed, round=rnd)
    torch.cuda.synchronize()
    for k in ("tokens", "q", "lse"):
        assert torch.equal(o[k], o2[k]), k
    return o, dbg


@pytest.mark.parametrize("B,Hd,V,T", [(4, 128, 1024, 1.0), (3, 192, 1000, 0.7), (1, 64, 512, 1.3),
                                      (40, 128, 2048, 1.0), (128, 64, 1024, 0.9),
                                      (32, 256, 8192, 1.0)])
def test_draft_small_shapes(B, Hd, V, T):
    h, W = make(B, Hd, V, seed=B + Hd + V)
    for rnd in range(3):
        check(h, W, T, seed=5, rnd=rnd, pos=rnd % 4)


def test_draft_full_size():
    """B=32, draft hidden 2048, V=128256 (the draft side of the lmhead workload)."""
    h, W = make(32, 2048, 128256, seed=11)
    for rnd in range(2):
        check(h, W, 1.0, seed=3, rnd=rnd, pos=1)


def test_draft_tokens_follow_q():
    """Over many rounds one row's tokens follow softmax of its logits (chi-square)."""
    h, W = make(1, 128, 64, seed=21, wstd=0.2)
    toks = []
    dbg = None
    for rnd in range(4000):
        o = sv.spec_lmhead_draft(h, W, pos=0, temperature=1.0, seed=1, round=rnd)
        toks.append(o["tokens"])
    dbg = torch.empty((1, 64), device="cuda")
    sv.spec_lmhead_draft(h, W, pos=0, temperature=1.0, seed=1, round=0, debug_logits=dbg)
    toks = torch.cat(toks).cpu().numpy()
    p = torch.softmax(dbg[0].double(), 0).cpu().numpy()
    obs = np.bincount(toks, minlength=64)
    keep = p * len(toks) >= 5
    assert chisq_pvalue(np.append(obs[keep], obs[~keep].sum()),
                        np.append(p[keep], p[~keep].sum())) > 1e-3


def test_draft_then_verify_chain():
    """Drafts drawn by spec_lmhead_draft feed spec_lmhead_verify: the verify's
    q(x) at the drafted tokens equals the draft's q(x) (same logits and T)."""
    B, gamma, V, Ht, Hd = 8, 3, 4096, 128, 128
    g = torch.Generator(device="cuda").manual_seed(31)
    h_t = torch.randn((B * (gamma + 1), Ht), generator=g, device="cuda").to(torch.bfloat16)
    W_t = (torch.randn((Ht, V), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    h_d = torch.randn((B * gamma, Hd), generator=g, device="cuda").to(torch.bfloat16)
    W_d = (torch.randn((Hd, V), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    hd3 = h_d.reshape(B, gamma, Hd)
    xt = torch.empty((B, gamma), dtype=torch.int32, device="cuda")
    qd = torch.empty((B, gamma), device="cuda")
    for i in range(gamma):
        o = sv.spec_lmhead_draft(hd3[:, i].contiguous(), W_d, pos=i, temperature=0.8, seed=4,
                                 round=9)
        xt[:, i] = o["tokens"]
        qd[:, i] = o["q"]
    v = sv.spec_lmhead_verify(h_t, W_t, h_d, W_d, xt, B=B, gamma=gamma, temperature=0.8,
                              seed=4, round=9)
    torch.cuda.synchronize()
    np.testing.assert_allclose(v["q"].cpu().numpy(), qd.cpu().numpy(), rtol=1e-4)


def _drafted_round(B, gamma, V, Ht, Hd, seed, T=1.0, rnd=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    h_t = torch.randn((B * (gamma + 1), Ht), generator=g, device="cuda").to(torch.bfloat16)
    W_t = (torch.randn((Ht, V), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    # a draft close to the target, so that rounds accept some drafts
    h_d = (h_t.reshape(B, gamma + 1, Ht)[:, :gamma].float() +
           0.05 * torch.randn((B, gamma, Hd), generator=g, device="cuda")).to(torch.bfloat16)
    W_d = (W_t.float() + 0.002 * torch.randn((Hd, V), generator=g, device="cuda")).to(
        torch.bfloat16)
    xt = torch.empty((B, gamma), dtype=torch.int32, device="cuda")
    lse = torch.empty((B, gamma), device="cuda")
    logit = torch.empty((B, gamma), device="cuda")
    zd = torch.empty((B, gamma, V), device="cuda")
    for i in range(gamma):
        dbg = torch.empty((B, V), device="cuda")
        o = sv.spec_lmhead_draft(h_d[:, i].contiguous(), W_d, pos=i, temperature=T, seed=seed,
                                 round=rnd, debug_logits=dbg)
        xt[:, i], lse[:, i], logit[:, i] = o["tokens"], o["lse"], o["logit"]
        zd[:, i] = dbg
    h_d = h_d.reshape(B * gamma, Hd).contiguous()
    return h_t, W_t, h_d, W_d, xt, lse, logit, zd


@pytest.mark.parametrize("B,gamma,V,Ht,Hd", [(8, 3, 4096, 128, 128), (32, 4, 16384, 256, 256)])
def test_drafted_verify_parity(B, gamma, V, Ht, Hd):
    """spec_lmhead_verify_drafted against the oracle on the logits both steps used:
    the target rows from the verify's debug output, the draft rows from the draft
    step's."""
    from tests._parity import assert_parity, to_np
    T = 0.9
    for rnd in range(2):
        h_t, W_t, h_d, W_d, xt, lse, logit, zd = _drafted_round(B, gamma, V, Ht, Hd, seed=41 + rnd,
                                                                 T=T, rnd=rnd)
        dbg = torch.full((B * (2 * gamma + 1), V), float("nan"), device="cuda")
        v = sv.spec_lmhead_verify_drafted(h_t, W_t, h_d, W_d, xt, lse, logit, B=B, gamma=gamma,
                                          temperature=T, seed=7, round=rnd, debug_logits=dbg)
        torch.cuda.synchronize()
        zt = dbg.reshape(B, 2 * gamma + 1, V)[:, :gamma + 1]
        assert torch.isfinite(zt).all()
        orc = oracle.spec_verify(zt.cpu().numpy(), zd.cpu().numpy(), xt.cpu().numpy(),
                                 temperature=T, seed=7, rnd=rnd, threads=8)
        assert_parity(to_np(v), orc, gamma, what=f"drafted verify B={B} round {rnd}")
        assert int(orc["counts"].max()) > 0  # some drafts accepted
        # the plain fused verify on the same inputs agrees
        w = sv.spec_lmhead_verify(h_t, W_t, h_d, W_d, xt, B=B, gamma=gamma, temperature=T, seed=7,
                                  round=rnd)
        torch.cuda.synchronize()
        assert torch.equal(w["counts"], v["counts"])
        assert torch.equal(w["tokens"], v["tokens"])
