"""Edge cases of the CUDA sampling path against the oracle (GPU)."""
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


def both(zt, zd, xt, T=1.0, rowT=None, seed=0, rnd=0, want_alpha=False):
    g = to_np(sv.spec_verify(zt, zd, xt, temperature=T, row_temperature=rowT, seed=seed,
                             round=rnd, want_alpha=want_alpha))
    o = oracle.spec_verify(wl.to_oracle(zt), wl.to_oracle(zd), xt.cpu().numpy(), temperature=T,
                           row_temperature=None if rowT is None else rowT.cpu().numpy(),
                           seed=seed, rnd=rnd, threads=THREADS, want_beta=want_alpha)
    return g, o


def rand_case(V, B=32, g=3, dtype=torch.float32, seed=0, spread=2.0, noise=0.7):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    zt = torch.randn((B, g + 1, V), generator=gen, device="cuda") * spread
    zd = zt[:, :g] + torch.randn((B, g, V), generator=gen, device="cuda") * noise
    zt, zd = zt.to(dtype).contiguous(), zd.to(dtype).contiguous()
    xt = wl.draw_from_logits(zd, 1.0, gen)
    return zt, zd, xt


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 16, 24, 31, 33, 1024, 2048, 2056, 4095, 4096,
                               4097, 4104, 8191, 8193, 16384, 24577])
def test_small_and_ragged_vocab(V, dtype):
    zt, zd, xt = rand_case(V, dtype=dtype, seed=V)
    for r in range(3):
        g, o = both(zt, zd, xt, seed=V, rnd=r, want_alpha=(r == 0))
        assert_parity(g, o, 3, what=f"V={V} {dtype} round {r}")
        if r == 0:
            np.testing.assert_allclose(g["alpha"], o["alpha"], rtol=1e-5, atol=1e-7)


def test_gamma_one_and_gamma_32():
    for gamma in (1, 32):
        zt, zd, xt = rand_case(1000, B=40, g=gamma, seed=gamma, noise=0.2)
        g, o = both(zt, zd, xt, seed=1, rnd=7)
        assert_parity(g, o, gamma, what=f"gamma={gamma}")
        assert g["counts"].max() <= gamma


def test_all_equal_rows_and_low_temperature():
    V, B, gm = 777, 16, 2
    zt = torch.zeros((B, gm + 1, V), device="cuda")
    zd = torch.zeros((B, gm, V), device="cuda")
    xt = torch.randint(0, V, (B, gm), device="cuda", dtype=torch.int32)
    g, o = both(zt, zd, xt, seed=4)
    assert_parity(g, o, gm, what="all-equal rows")
    assert np.all(g["counts"] == gm)  # p == q: every draft accepted
    zt2, zd2, xt2 = rand_case(500, B=16, g=2, seed=9)
    g, o = both(zt2, zd2, xt2, T=0.05, seed=4)
    assert_parity(g, o, 2, what="T=0.05")


def test_minus_inf_masks_and_residual_repair():
    V, B, gm = 3000, 24, 4
    zt, zd, xt = rand_case(V, B=B, g=gm, seed=13, noise=1.5)
    gen = torch.Generator(device="cuda").manual_seed(1)
    mask = torch.rand((B, gm, V), generator=gen, device="cuda") < 0.2
    zd = zd.masked_fill(mask, float("-inf")).contiguous()
    xt = wl.draw_from_logits(zd, 1.0, gen)
    for r in range(4):
        g, o = both(zt, zd, xt, seed=2, rnd=r)
        assert_parity(g, o, gm, what=f"-inf masks round {r}")


def test_forced_empty_residual_and_empty_rows():
    V, B = 40, 8
    row = torch.randn(V, device="cuda")
    row[5] = float("-inf")
    zt = row.expand(B, 2, V).contiguous()
    zd = row.expand(B, 1, V).contiguous()
    xt = torch.full((B, 1), 5, dtype=torch.int32, device="cuda")  # p = q = 0 at the draft
    g, o = both(zt, zd, xt, seed=6)
    assert_parity(g, o, 1, what="forced empty residual")
    assert np.all(g["flags"] & sv.FLAG_RESIDUAL_FALLBACK)
    # a bonus row with no finite logit, and a draft token out of range
    zt2 = torch.zeros((2, 3, 16), device="cuda")
    zt2[0, 2] = float("-inf")
    zd2 = torch.zeros((2, 2, 16), device="cuda")
    xt2 = torch.tensor([[1, 2], [1, 99]], dtype=torch.int32, device="cuda")
    g, o = both(zt2, zd2, xt2, seed=1)
    assert_parity(g, o, 2, what="empty bonus row / bad token")
    assert g["flags"][0] & sv.FLAG_ZERO_MASS and g["flags"][1] & sv.FLAG_BAD_TOKEN


def test_q_zero_at_draft_and_nonfinite_flag():
    V = 64
    zt = torch.zeros((4, 2, V), device="cuda")
    zd = torch.zeros((4, 1, V), device="cuda")
    zd[:, 0, 3] = float("-inf")
    xt = torch.full((4, 1), 3, dtype=torch.int32, device="cuda")
    g, o = both(zt, zd, xt, seed=1)
    assert_parity(g, o, 1, what="q(x)=0")
    assert np.all(g["counts"] == 1) and np.all(g["flags"] & sv.FLAG_NONFINITE)
    zt[1, 0, 7] = float("nan")
    g = to_np(sv.spec_verify(zt, zd, xt, seed=1))
    assert g["flags"][1] & sv.FLAG_NONFINITE
    assert g["tokens"].max() < V and g["tokens"].min() >= -1


def test_per_row_temperature():
    zt, zd, xt = rand_case(5000, B=32, g=3, dtype=torch.bfloat16, seed=21)
    T = torch.linspace(0.3, 2.0, 32, device="cuda")
    g, o = both(zt, zd, xt, T=1.0, rowT=T, seed=3)
    assert_parity(g, o, 3, what="per-row T")


def test_workspace_reuse_and_determinism():
    zt, zd, xt = rand_case(20000, B=16, g=4, dtype=torch.bfloat16, seed=31)
    ws = sv.alloc_workspace(16, 4, 20000, 0)
    a = to_np(sv.spec_verify(zt, zd, xt, seed=9, round=3, workspace=ws))
    b = to_np(sv.spec_verify(zt, zd, xt, seed=9, round=3, workspace=ws))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = sv.spec_verify(zt, zd, xt, seed=9, round=3, stream=s)
    s.synchronize()
    c = to_np(c)
    for k in ("tokens", "counts", "p", "q", "flags"):
        np.testing.assert_array_equal(a[k], b[k])
        np.testing.assert_array_equal(a[k], c[k])
    # the workspace needs no initial contents: garbage in it changes nothing
    ws.fill_(0xFF)
    d = to_np(sv.spec_verify(zt, zd, xt, seed=9, round=3, workspace=ws))
    for k in ("tokens", "counts", "p", "q", "flags"):
        np.testing.assert_array_equal(a[k], d[k])


def test_misaligned_pointer_rejected():
    zt, zd, xt = rand_case(64, B=2, g=1, seed=1)
    flat = torch.zeros(zt.numel() + 1, device="cuda")
    zt_mis = flat[1:].view_as(zt)  # 4-byte offset
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_verify(zt_mis, zd, xt)
    assert e.value.status == -3


@pytest.mark.parametrize("V,dtype", [(131072, torch.bfloat16), (131080, torch.bfloat16),
                                     (262147, torch.float32)])
def test_large_vocab(V, dtype):
    """Long rows: many race slices per batch row (a ragged last slice), the
    separate-kernel path for a row length that is not a multiple of 16 bytes."""
    zt, zd, xt = rand_case(V, B=8, g=2, dtype=dtype, seed=V % 1000)
    for r in range(3):
        g, o = both(zt, zd, xt, seed=5, rnd=r)
        assert_parity(g, o, 2, what=f"V={V} {dtype} round {r}")


def test_forced_empty_residual_long_row():
    """The empty-residual fallback on a row longer than one search round."""
    V, B = 140000, 4
    gen = torch.Generator(device="cuda").manual_seed(3)
    row = torch.randn(V, generator=gen, device="cuda")
    row[11] = float("-inf")
    zt = row.expand(B, 2, V).contiguous()
    zd = row.expand(B, 1, V).contiguous()
    xt = torch.full((B, 1), 11, dtype=torch.int32, device="cuda")
    for r in range(2):
        g, o = both(zt, zd, xt, seed=8, rnd=r)
        assert_parity(g, o, 1, what=f"forced empty residual, V={V}")
        assert np.all(g["flags"] & sv.FLAG_RESIDUAL_FALLBACK)


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 6000), (torch.float32, 6000),
                                     (torch.bfloat16, 6001), (torch.bfloat16, 128256)])
def test_outputs_do_not_depend_on_addresses(dtype, V):
    """The same logits at three places in memory (16-byte aligned views starting
    at different offsets within a 4 KB block) give bit-identical tokens, counts,
    p, q, alpha and flags: the sweep cuts every row from its own start, so no sum
    depends on where the row sits.  V = 6001 (bf16) takes the generic sweep (rows
    not a multiple of 16 bytes), the others the vector sweep."""
    B, g = 8, 3
    zt0, zd0, xt = rand_case(V, B=B, g=g, dtype=dtype, seed=V)
    esz = 4 if dtype == torch.float32 else 2
    outs = []
    for off_t, off_d in ((0, 0), (8 * 16 // esz, 24 * 16 // esz), (2040 * 2 // esz, 16 // esz)):
        bt = torch.empty(zt0.numel() + off_t, dtype=dtype, device="cuda")
        bd = torch.empty(zd0.numel() + off_d, dtype=dtype, device="cuda")
        zt = bt[off_t:].view(zt0.shape)
        zd = bd[off_d:].view(zd0.shape)
        zt.copy_(zt0)
        zd.copy_(zd0)
        assert zt.data_ptr() % 16 == 0 and zd.data_ptr() % 16 == 0
        rounds = []
        for r in range(3):
            gg = to_np(sv.spec_verify(zt, zd, xt, seed=3, round=r, want_alpha=(r == 0)))
            rounds.append(gg)
        outs.append(rounds)
        del bt, bd
    for rounds in outs[1:]:
        for r in range(3):
            for k in ("tokens", "counts", "p", "q", "flags") + (("alpha",) if r == 0 else ()):
                np.testing.assert_array_equal(rounds[r][k], outs[0][r][k], err_msg=f"{k} r={r}")
    # and the first placement against the oracle
    for r in range(3):
        o = oracle.spec_verify(wl.to_oracle(zt0), wl.to_oracle(zd0), xt.cpu().numpy(), seed=3,
                               rnd=r, threads=THREADS)
        assert_parity(outs[0][r], o, g, what=f"addresses {dtype} V={V} round {r}")
