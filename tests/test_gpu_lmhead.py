"""Fused LM heads + verify (spec_lmhead_verify) on the GPU.

Rules for the fused path: its logits (returned through debug_logits) are within
2e-2 absolute of an fp32 reference of h W, and of the oracle's double-precision
product on sampled columns; its decisions are compared with the oracle run on
those identical logits (tests/_parity.py rules).  A call without debug_logits
gives the same outputs as one with it.
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
LOGIT_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.backends.cuda.matmul.allow_tf32 = False
    sv.load()


def make_case(B, gamma, V, Ht, Hd, seed, mode="independent", wstd=0.02):
    """h ~ N(0,1), W ~ N(0, wstd^2) in bf16; draft tokens drawn from the draft's
    own logits.  mode 'shared': the draft is the target (p = q, every draft
    accepted); 'close': the draft is a perturbed copy of the target."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    dev = "cuda"
    h_t = torch.randn((B * (gamma + 1), Ht), generator=g, device=dev).to(torch.bfloat16)
    W_t = (torch.randn((Ht, V), generator=g, device=dev) * wstd).to(torch.bfloat16)
    pos = torch.arange(B * (gamma + 1), device=dev) % (gamma + 1) < gamma
    if mode == "shared":
        assert Hd == Ht
        h_d = h_t[pos].contiguous()
        W_d = W_t.clone()
    elif mode == "close":
        assert Hd == Ht
        h_d = (h_t[pos].float() + 0.05 * torch.randn((B * gamma, Hd), generator=g,
                                                      device=dev)).to(torch.bfloat16)
        W_d = (W_t.float() + 0.1 * wstd * torch.randn((Hd, V), generator=g,
                                                       device=dev)).to(torch.bfloat16)
    else:
        h_d = torch.randn((B * gamma, Hd), generator=g, device=dev).to(torch.bfloat16)
        W_d = (torch.randn((Hd, V), generator=g, device=dev) * wstd).to(torch.bfloat16)
    zd = (h_d.float() @ W_d.float()).reshape(B, gamma, V)
    xt = wl.draw_from_logits(zd, 1.0, g)
    return h_t, W_t, h_d.contiguous(), W_d.contiguous(), xt


def run_lm(case, B, gamma, T=1.0, seed=0, rnd=0, debug=True):
    h_t, W_t, h_d, W_d, xt = case
    V = W_t.shape[1]
    dbg = torch.full((B * (2 * gamma + 1), V), float("nan"), device="cuda") if debug else None
    o = sv.spec_lmhead_verify(h_t, W_t, h_d, W_d, xt, B=B, gamma=gamma, temperature=T,
                              seed=seed, round=rnd, debug_logits=dbg)
    torch.cuda.synchronize()
    return to_np(o), dbg


def split_logits(dbg, B, gamma):
    V = dbg.shape[1]
    z = dbg.reshape(B, 2 * gamma + 1, V)
    return z[:, :gamma + 1].contiguous(), z[:, gamma + 1:].contiguous()


def check_logits(case, dbg, B, gamma, ncols=64, seed=0):
    h_t, W_t, h_d, W_d, _ = case
    V = W_t.shape[1]
    zt, zd = split_logits(dbg, B, gamma)
    ref_t = (h_t.float() @ W_t.float()).reshape(B, gamma + 1, V)
    ref_d = (h_d.float() @ W_d.float()).reshape(B, gamma, V)
    assert torch.isfinite(dbg).all(), "debug logits not fully written"
    et = (zt - ref_t).abs().max().item()
    ed = (zd - ref_d).abs().max().item()
    assert et <= LOGIT_TOL and ed <= LOGIT_TOL, (et, ed)
    # the oracle's double-precision product on sampled columns (and rows)
    rng = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([rng.integers(0, V, ncols), [0, V - 1]]))
    rt = np.unique(rng.integers(0, h_t.shape[0], 8))
    rd = np.unique(rng.integers(0, h_d.shape[0], 8))
    ot = oracle.lmhead_logits(wl.bf16_bits(h_t[rt]), wl.bf16_bits(W_t), cols=cols)
    od = oracle.lmhead_logits(wl.bf16_bits(h_d[rd]), wl.bf16_bits(W_d), cols=cols)
    gt = zt.reshape(-1, V)[rt][:, cols].cpu().numpy()
    gd = zd.reshape(-1, V)[rd][:, cols].cpu().numpy()
    assert np.abs(gt - ot).max() <= LOGIT_TOL
    assert np.abs(gd - od).max() <= LOGIT_TOL
    return et, ed


def check_decisions(gpu, dbg, xt, B, gamma, T, seed, rnd, what):
    zt, zd = split_logits(dbg, B, gamma)
    orc = oracle.spec_verify(zt.cpu().numpy(), zd.cpu().numpy(), xt.cpu().numpy(),
                             temperature=T, seed=seed, rnd=rnd, threads=THREADS)
    return assert_parity(gpu, orc, gamma, what=what), orc


def full_check(B, gamma, V, Ht, Hd, seed, mode="independent", T=1.0, rounds=(0, 1)):
    case = make_case(B, gamma, V, Ht, Hd, seed, mode)
    stats = []
    for rnd in rounds:
        gpu, dbg = run_lm(case, B, gamma, T=T, seed=seed, rnd=rnd)
        if rnd == rounds[0]:
            check_logits(case, dbg, B, gamma, seed=seed)
        _, orc = check_decisions(gpu, dbg, case[4], B, gamma, T, seed, rnd,
                                 f"lmhead B={B} g={gamma} V={V} {mode} round {rnd}")
        # the same call without the debug output gives the same result
        gpu2, _ = run_lm(case, B, gamma, T=T, seed=seed, rnd=rnd, debug=False)
        for k in ("tokens", "counts", "flags", "p", "q"):
            np.testing.assert_array_equal(gpu[k], gpu2[k], err_msg=k)
        stats.append(orc)
    return stats


def test_lmhead_small():
    stats = full_check(2, 2, 1024, 128, 128, seed=11, rounds=(0, 1, 2, 3))
    assert any(int(o["counts"].min()) < 2 for o in stats)  # rejections (pass 2) happened


def test_lmhead_ragged_vocab_and_hidden():
    # V = 1000: the last 128-entry tile holds 104 entries; hidden 192 / 64
    full_check(3, 3, 1000, 192, 64, seed=12, rounds=(0, 1, 2))


def test_lmhead_two_row_tiles():
    # 200 target rows and 160 draft rows: two 128-row tiles on both sides
    full_check(40, 4, 2048, 128, 128, seed=13)


def test_lmhead_max_rows():
    # B*(gamma+1) = 256 target rows, 128 draft rows, 128 compact rows possible
    full_check(128, 1, 512, 64, 64, seed=14)


def test_lmhead_all_accepted_bonus_path():
    stats = full_check(4, 3, 4096, 256, 256, seed=15, mode="shared", rounds=(0, 1, 2))
    for o in stats:
        assert np.all(o["counts"] == 3)  # p = q: every draft accepted, bonus from p_gamma


def test_lmhead_close_draft_mixed_outcomes():
    stats = full_check(16, 4, 8192, 256, 256, seed=16, mode="close", rounds=(0, 1, 2, 3))
    counts = np.concatenate([o["counts"] for o in stats])
    assert counts.min() < 4 and counts.max() == 4


def test_lmhead_temperature():
    full_check(8, 3, 4096, 128, 128, seed=17, T=0.7, rounds=(0, 1))


def test_lmhead_bad_tokens():
    B, gamma, V = 4, 2, 1024
    case = list(make_case(B, gamma, V, 128, 128, seed=18))
    xt = case[4].clone()
    xt[0, 0] = -1
    xt[1, 1] = V
    case[4] = xt
    gpu, dbg = run_lm(tuple(case), B, gamma, seed=3, rnd=5)
    check_decisions(gpu, dbg, xt, B, gamma, 1.0, 3, 5, "lmhead bad tokens")
    assert gpu["flags"][0] & 16 and gpu["flags"][1] & 16


def test_lmhead_config5_full_size():
    """B=32, gamma=4, V=128256, target hidden 4096, draft hidden 2048."""
    B, gamma, V, Ht, Hd = 32, 4, 128256, 4096, 2048
    case = make_case(B, gamma, V, Ht, Hd, seed=1005)
    for rnd in (0, 1):
        gpu, dbg = run_lm(case, B, gamma, seed=7, rnd=rnd)
        if rnd == 0:
            et, ed = check_logits(case, dbg, B, gamma, ncols=32)
        check_decisions(gpu, dbg, case[4], B, gamma, 1.0, 7, rnd, f"config 5 round {rnd}")
        gpu2, _ = run_lm(case, B, gamma, seed=7, rnd=rnd, debug=False)
        for k in ("tokens", "counts", "flags"):
            np.testing.assert_array_equal(gpu[k], gpu2[k], err_msg=k)
