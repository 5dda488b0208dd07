"""Parity of the CUDA path (through the C ABI) with the oracle, on the GPU.

Inputs are the seeded synthetic workloads (speculative_decoding_verification_21_gb300.workloads),
generated on the device and copied to the host for the oracle.  Rules are in
tests/_parity.py.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import speculative_decoding_verification_21_gb300 as sv
from speculative_decoding_verification_21_gb300 import workloads as wl
from tests._helpers import chisq_pvalue
from tests._parity import assert_parity, to_np

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


def test_sample_b1_fp32_many_rounds():
    near = dec = 0
    for r in range(0, 400):
        w = wl.sample_b1(seed=5000 + r // 4)  # fresh logits every 4 rounds
        gpu, orc = run_both(w, seed=0, rnd=r)
        n, d = assert_parity(gpu, orc, w.gamma, what=f"sample_b1 round {r}")
        near, dec = near + n, dec + d
    assert near <= 1e-4 * dec


@pytest.mark.parametrize("sigma", [0.25, 1.0, 4.0])
def test_sample_b64_full(sigma):
    w = wl.sample_b64(sigma=sigma)
    near = dec = 0
    for r in range(3):
        gpu, orc = run_both(w, seed=0, rnd=r, want_alpha=(r == 0))
        n, d = assert_parity(gpu, orc, w.gamma, what=f"sample_b64 sigma={sigma} round {r}")
        near, dec = near + n, dec + d
        if r == 0:
            np.testing.assert_allclose(gpu["alpha"], orc["alpha"], rtol=1e-5)
    assert near <= 1e-4 * max(dec, 1e4)


@pytest.mark.parametrize("lenience", [0.5, 0.1])
def test_sample_b64_lenience(lenience):
    """Lenient comparison u <= p/(l q) against the oracle's, and more acceptances
    than the exact round on the same inputs and uniforms."""
    w = wl.sample_b64(sigma=1.0)
    near = dec = 0
    for r in range(2):
        gpu, orc = run_both(w, seed=0, rnd=r, lenience=lenience)
        n, d = assert_parity(gpu, orc, w.gamma, what=f"sample_b64 lenience={lenience} round {r}")
        near, dec = near + n, dec + d
        exact, _ = run_both(w, seed=0, rnd=r, rows=[0])
        assert np.all(gpu["counts"] >= exact["counts"])
        assert gpu["counts"].sum() > exact["counts"].sum()
    assert near <= 1e-4 * max(dec, 1e4)


def test_sample_b256_sampled_rows():
    w = wl.sample_b256()
    rng = np.random.default_rng(0)
    masked = w.extra["masked_rows"].any(dim=1).cpu().numpy()
    rows = sorted(set(rng.choice(w.B, 12, replace=False).tolist()) |
                  set(np.nonzero(masked)[0][:4].tolist()))
    for r in range(2):
        gpu, orc = run_both(w, seed=11, rnd=r, rows=rows)
        assert_parity(gpu, orc, w.gamma, rows=rows, what=f"sample_b256 round {r}")


def test_greedy_b64_full_bit_exact():
    w = wl.greedy_b64()
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
    tgt = torch.from_numpy(oracle.spec_verify_greedy(
        wl.to_oracle(zt), np.zeros((B, g), np.int32))["tokens"][:, :1])
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
    del tgt
