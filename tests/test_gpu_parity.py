"""Parity of the CUDA path (through the C ABI) with the oracle, on the GPU, at
the workloads' stated scale.

Inputs are the seeded synthetic workloads (speculative_decoding_verification_21_gb300.workloads),
generated on the device and copied to the host for the oracle.  Rules are in
tests/_parity.py; each sampling workload reports its decision count and its
near-ties in the session summary.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_21_gb300 as sv
from speculative_decoding_verification_21_gb300 import workloads as wl
from tests._helpers import chisq_pvalue
from tests._parity import NEAR_TIE_RATE, assert_parity, near_ties, record, to_np

pytestmark = pytest.mark.gpu
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()


def run_both(w, seed=0, rnd=0, rows=None, want_alpha=False, lenience=1.0):
    g = sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature,
                       row_temperature=w.row_temperature, seed=seed, round=rnd,
                       want_alpha=want_alpha, lenience=lenience)
    torch.cuda.synchronize()
    gpu = to_np(g)
    rowT = None if w.row_temperature is None else w.row_temperature.cpu().numpy()
    orc = oracle.spec_verify(wl.to_oracle(w.zt), wl.to_oracle(w.zd), w.xt.cpu().numpy(),
                             temperature=w.temperature, row_temperature=rowT, seed=seed, rnd=rnd,
                             rows=rows, threads=THREADS, want_beta=want_alpha,
                             lenience=lenience)
    return gpu, orc


class Tally:
    def __init__(self):
        self.dec = self.near = self.near_o = 0

    def add(self, gpu, orc, gamma, what, rows=None):
        n, d = assert_parity(gpu, orc, gamma, rows=rows, what=what)
        self.dec += d
        self.near += n
        self.near_o += near_ties(orc, gamma, rows)

    def close(self, what):
        record(what, self.dec, self.near, self.near_o)
        assert self.dec >= 10_000, f"{what}: only {self.dec} decisions"
        assert self.near <= NEAR_TIE_RATE * self.dec, f"{what}: {self.near} near-ties"


def test_three_token_example_gpu():
    """The lihaoran.work essay's three-token example through the GPU path: the
    emitted token is distributed as p = (0.6, 0.3, 0.1) and every decision
    matches the oracle."""
    w = wl.three_token(200_000)
    gpu, orc = run_both(w, seed=3, rnd=1)
    assert_parity(gpu, orc, 1, what="three-token")
    counts = np.bincount(gpu["tokens"][:, 0], minlength=3)
    assert chisq_pvalue(counts, [0.6, 0.3, 0.1]) > 1e-3
    acc = (gpu["counts"] == 1).mean()
    assert abs(acc - 0.6) < 4 * np.sqrt(0.24 / 200_000)


def test_sample_b1_fp32_rounds():
    """B=1, gamma=4, V=32000 fp32, fresh logits every round: the stated 1000
    rounds, then on to 10^4 decisions."""
    t = Tally()
    r = 0
    while r < 1000 or t.dec < 10_000:
        w = wl.sample_b1(seed=5000 + r)
        gpu, orc = run_both(w, seed=0, rnd=r)
        t.add(gpu, orc, w.gamma, f"sample_b1 round {r}")
        r += 1
    t.close(f"sample_b1 (B=1, gamma=4, V=32000, fp32; {r} rounds)")


@pytest.mark.parametrize("sigma", [0.25, 1.0, 4.0])
def test_sample_b64_100_rounds(sigma):
    """B=64, gamma=4, V=128256 bf16, T=0.8: 100 rounds per draft-noise level."""
    w = wl.sample_b64(sigma=sigma)
    t = Tally()
    for r in range(100):
        gpu, orc = run_both(w, seed=0, rnd=r, want_alpha=(r == 0))
        t.add(gpu, orc, w.gamma, f"sample_b64 sigma={sigma} round {r}")
        if r == 0:
            np.testing.assert_allclose(gpu["alpha"], orc["alpha"], rtol=1e-5)
    t.close(f"sample_b64 sigma={sigma} (100 rounds)")


def test_sample_b256_all_rows_20_rounds():
    """B=256, gamma=8, V=152064 bf16, per-row T and noise, -inf masks: every batch
    row for 20 rounds."""
    w = wl.sample_b256()
    t = Tally()
    assert w.extra["masked_rows"].any()
    for r in range(20):
        gpu, orc = run_both(w, seed=11, rnd=r)
        t.add(gpu, orc, w.gamma, f"sample_b256 round {r}")
    t.close("sample_b256 (all 256 rows, 20 rounds)")


@pytest.mark.parametrize("lenience", [0.5, 0.1])
def test_sample_b64_lenience(lenience):
    """Lenient comparison u <= p/(l q) against the oracle's, and more acceptances
    than the exact round on the same inputs and uniforms."""
    w = wl.sample_b64(sigma=1.0)
    for r in range(2):
        gpu, orc = run_both(w, seed=0, rnd=r, lenience=lenience)
        assert_parity(gpu, orc, w.gamma, what=f"sample_b64 lenience={lenience} round {r}")
        exact, _ = run_both(w, seed=0, rnd=r, rows=[0])
        assert np.all(gpu["counts"] >= exact["counts"])
        assert gpu["counts"].sum() > exact["counts"].sum()


def test_greedy_b64_full_bit_exact():
    w = wl.greedy_b64()
    for rnd in range(3):
        g = sv.spec_verify_greedy(w.zt, w.xt)
        torch.cuda.synchronize()
        o = oracle.spec_verify_greedy(wl.to_oracle(w.zt), w.xt.cpu().numpy())
        np.testing.assert_array_equal(g["tokens"].cpu().numpy(), o["tokens"])
        np.testing.assert_array_equal(g["counts"].cpu().numpy(), o["counts"])
    # the workload exercises both outcomes
    c = o["counts"]
    assert (c == 0).any() and (c > 0).any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 31, 33, 8191, 8193, 20011])
def test_greedy_small_and_ragged(V, dtype):
    gen = torch.Generator(device="cuda").manual_seed(V)
    B, g = 24, 3
    # small integers: many exact ties; plus -inf and NaN entries
    zt = torch.randint(-3, 4, (B, g + 1, V), generator=gen, device="cuda").float()
    zt[torch.rand(zt.shape, generator=gen, device="cuda") < 0.05] = float("-inf")
    zt[torch.rand(zt.shape, generator=gen, device="cuda") < 0.02] = float("nan")
    zt[0] = float("-inf")
    zt = zt.to(torch.bfloat16) if dtype == "bf16" else zt
    xt = torch.randint(0, V, (B, g), generator=gen, device="cuda").to(torch.int32)
    ref_t = []
    for i in range(g):  # copy some target argmaxes so prefixes match
        o = oracle.spec_verify_greedy(wl.to_oracle(zt[:, i:i + 2].contiguous()),
                                      np.zeros((B, 1), np.int32))
        ref_t.append(o["tokens"][:, 0])
    ref_t = torch.tensor(np.stack(ref_t, 1), device="cuda", dtype=torch.int32)
    keep = torch.rand((B, g), generator=gen, device="cuda") < 0.7
    xt = torch.where(keep, ref_t, xt).contiguous()
    out = sv.spec_verify_greedy(zt.contiguous(), xt)
    torch.cuda.synchronize()
    o = oracle.spec_verify_greedy(wl.to_oracle(zt), xt.cpu().numpy())
    np.testing.assert_array_equal(out["tokens"].cpu().numpy(), o["tokens"])
    np.testing.assert_array_equal(out["counts"].cpu().numpy(), o["counts"])
