"""Greedy pins (brute force, T->0 limit) and edge cases of the oracle."""
import numpy as np
import pytest

import oracle
from tests._helpers import logits_from_probs


def _brute_greedy(zt, xt):
    B, g1, V = zt.shape
    g = g1 - 1
    toks = np.full((B, g1), -1, np.int32)
    cnt = np.zeros(B, np.int32)
    for b in range(B):
        tgt = []
        for i in range(g1):
            best, arg = None, 0
            for v in range(V):
                z = float(zt[b, i, v])
                if z != z:
                    z = -np.inf
                if best is None or z > best:
                    best, arg = z, v
            tgt.append(arg)
        n = g
        for i in range(g):
            if xt[b, i] != tgt[i]:
                n = i
                break
        toks[b, :n] = xt[b, :n]
        toks[b, n] = tgt[n]
        cnt[b] = n
    return toks, cnt


def _bf16_bits(x):
    """Round-to-nearest-even float32 -> bf16 bit patterns (uint16)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


@pytest.mark.parametrize("V,g,seed", [(1, 1, 0), (2, 3, 1), (7, 2, 2), (8, 4, 3), (9, 1, 4)])
def test_greedy_bruteforce_ties(V, g, seed):
    rng = np.random.default_rng(seed)
    B = 64
    # small integer logits -> many exact ties, plus -inf and NaN entries
    zt = rng.integers(-2, 3, (B, g + 1, V)).astype(np.float32)
    zt[rng.random(zt.shape) < 0.1] = -np.inf
    zt[rng.random(zt.shape) < 0.05] = np.nan
    zt[0] = -np.inf  # an all -inf batch row: argmax is index 0
    xt = rng.integers(0, V, (B, g)).astype(np.int32)
    # make many prefixes match: copy the brute-force target argmaxes
    tgt = np.array([[_brute_greedy(zt[b:b + 1, i:i + 1], np.zeros((1, 0), np.int32))[0][0, 0]
                     for i in range(g)] for b in range(B)], np.int32)
    for b in range(B // 2):
        k = int(rng.integers(0, g + 1))
        xt[b, :k] = tgt[b, :k]
    ref_t, ref_c = _brute_greedy(zt, xt)
    out = oracle.spec_verify_greedy(zt, xt)
    np.testing.assert_array_equal(out["tokens"], ref_t)
    np.testing.assert_array_equal(out["counts"], ref_c)
    # bf16 path gives the same answer on bf16-representable values
    out16 = oracle.spec_verify_greedy(_bf16_bits(zt), xt)
    np.testing.assert_array_equal(out16["tokens"], ref_t)


def test_sampling_tends_to_greedy_as_T_goes_to_zero():
    """'Fast Inference ...', 'Speculative sampling: the accept/reject rule': at low
    temperature both distributions collapse on their argmax and the rule becomes
    argmax decoding with a verify step."""
    rng = np.random.default_rng(3)
    B, g, V = 200, 4, 50
    # distinct logits (gaps >= 0.01) so argmaxes are unique
    zt = np.stack([rng.permutation(V) for _ in range(B * (g + 1))]).reshape(B, g + 1, V)
    zt = (zt * 0.01).astype(np.float32)
    zd = zt[:, :g].copy()
    swap = rng.random((B, g)) < 0.3  # draft argmax differs at some positions
    for b, i in zip(*np.nonzero(swap)):
        zd[b, i] = np.roll(zd[b, i], 1)
    xt = zd.argmax(axis=2).astype(np.int32)
    greedy = oracle.spec_verify_greedy(zt, xt)
    samp = oracle.spec_verify(zt, zd, xt, temperature=1e-4, seed=5)
    np.testing.assert_array_equal(samp["tokens"], greedy["tokens"])
    np.testing.assert_array_equal(samp["counts"], greedy["counts"])


def test_edge_empty_bonus_row_and_bad_token():
    V, g = 5, 2
    zt = np.zeros((2, g + 1, V), np.float32)
    zd = np.zeros((2, g, V), np.float32)
    zt[0, g] = -np.inf  # bonus row has no finite logit
    xt = np.array([[1, 2], [1, 7]], np.int32)  # row 1: token 7 is out of range
    out = oracle.spec_verify(zt, zd, xt, seed=1)
    assert out["counts"][0] == g and out["tokens"][0, g] == 0
    assert out["flags"][0] & oracle.FLAG_ZERO_MASS
    assert out["counts"][1] == 1 and out["flags"][1] & oracle.FLAG_BAD_TOKEN
    assert np.all(out["tokens"][1] >= -1) and out["tokens"][1, 1] < V


def test_edge_forced_empty_residual_falls_back_to_p():
    """Identical target/draft rows with the draft token on a -inf logit: p = q = 0
    there, so the test rejects (0/0) while max(0, p - q) has no mass."""
    V, n = 6, 200_000
    row = logits_from_probs([0.3, 0.2, 0.1, 0.25, 0.15, 0.0])
    zt = np.broadcast_to(np.stack([row, row]), (n, 2, V)).copy()
    zd = np.broadcast_to(row, (n, 1, V)).copy()
    xt = np.full((n, 1), 5, np.int32)
    out = oracle.spec_verify(zt, zd, xt, seed=2)
    assert np.all(out["counts"] == 0)
    assert np.all(out["flags"] & oracle.FLAG_RESIDUAL_FALLBACK)
    from tests._helpers import chisq_pvalue
    assert chisq_pvalue(np.bincount(out["tokens"][:, 0], minlength=V)[:5],
                        [0.3, 0.2, 0.1, 0.25, 0.15]) > 1e-3


def test_edge_q_zero_at_draft_accepts_and_flags():
    V = 3
    zt = np.broadcast_to(logits_from_probs([0.5, 0.3, 0.2]), (4, 2, V)).copy()
    zd = np.broadcast_to(logits_from_probs([0.0, 0.6, 0.4]), (4, 1, V)).copy()
    xt = np.zeros((4, 1), np.int32)  # the draft token has q = 0, p > 0
    out = oracle.spec_verify(zt, zd, xt, seed=3)
    assert np.all(out["counts"] == 1)
    assert np.all(out["flags"] & oracle.FLAG_NONFINITE)
    assert np.all(np.isinf(out["ratio"][:, 0]))


def test_edge_nonfinite_logits_flagged():
    V = 4
    zt = np.zeros((1, 2, V), np.float32)
    zd = np.zeros((1, 1, V), np.float32)
    zt[0, 0, 2] = np.nan
    out = oracle.spec_verify(zt, zd, np.zeros((1, 1), np.int32), seed=3)
    assert out["flags"][0] & oracle.FLAG_NONFINITE
    assert -1 <= out["tokens"][0].min() and out["tokens"][0].max() < V


def test_edge_v1_and_arguments():
    zt = np.zeros((3, 2, 1), np.float32)
    zd = np.zeros((3, 1, 1), np.float32)
    out = oracle.spec_verify(zt, zd, np.zeros((3, 1), np.int32))
    np.testing.assert_array_equal(out["tokens"], np.zeros((3, 2), np.int32))
    np.testing.assert_array_equal(out["counts"], [1, 1, 1])
    with pytest.raises(ValueError):
        oracle.spec_verify(np.zeros((1, 1, 4), np.float32), np.zeros((1, 0, 4), np.float32),
                           np.zeros((1, 0), np.int32))
