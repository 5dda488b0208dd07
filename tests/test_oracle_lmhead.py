"""Pins of the oracle's LM-head reference, logits = h W (bf16 inputs, double
accumulation), against closed forms ("Fast Inference from Transformers via
Speculative Decoding", section "The loop ...": the logits are the final
projection of the model pass).  Each case has an exact answer that does not
come from a matrix product routine: selection by unit vectors (catches a
transposed operand or a wrong row stride), arithmetic-series sums, a rank-one
product of small integers, and column subsets in a given order."""
import numpy as np

import oracle


def bf16(a):
    """float array of bf16-exact values -> uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "values must be bf16-exact"
    return (bits >> 16).astype(np.uint16)


def test_unit_vectors_select_rows_of_W():
    H, V = 8, 24
    rng = np.random.default_rng(0)
    W = (rng.integers(-64, 64, size=(H, V)) / 8.0).astype(np.float32)
    h = np.zeros((3, H), np.float32)
    h[0, 0] = 1.0
    h[1, 5] = 1.0
    h[2, 7] = -2.0
    out = oracle.lmhead_logits(bf16(h), bf16(W))
    assert out.shape == (3, V)
    np.testing.assert_array_equal(out[0], W[0])
    np.testing.assert_array_equal(out[1], W[5])
    np.testing.assert_array_equal(out[2], -2.0 * W[7])


def test_arithmetic_series():
    # h = all ones, W[k][v] = k + v: logit[v] = H(H-1)/2 + H v
    H, V = 64, 40
    k = np.arange(H, dtype=np.float32)[:, None]
    v = np.arange(V, dtype=np.float32)[None, :]
    W = k + v
    h = np.ones((2, H), np.float32)
    out = oracle.lmhead_logits(bf16(h), bf16(W))
    expect = H * (H - 1) / 2 + H * np.arange(V)
    np.testing.assert_array_equal(out[0], expect)
    np.testing.assert_array_equal(out[1], expect)


def test_rank_one_integers():
    # h[m][k] = a_m, W[k][v] = c_k b_v: logit = a_m b_v sum_k c_k
    a = np.array([1, -2, 3], np.float32)
    b = np.array([2, 0, -1, 5, 7], np.float32)
    c = np.array([1, 2, 3, 4, -1, -2, 0, 5], np.float32)  # sum 12
    h = np.repeat(a[:, None], c.size, axis=1)
    W = c[:, None] * b[None, :]
    out = oracle.lmhead_logits(bf16(h), bf16(W))
    np.testing.assert_array_equal(out, 12.0 * a[:, None] * b[None, :])


def test_alternating_signs_cancel():
    H, V = 32, 6
    h = np.where(np.arange(H) % 2 == 0, 1.0, -1.0).astype(np.float32)[None, :]
    W = np.full((H, V), 3.0, np.float32)
    out = oracle.lmhead_logits(bf16(h), bf16(W))
    np.testing.assert_array_equal(out, np.zeros((1, V)))


def test_column_subset_in_given_order():
    H, V = 8, 16
    W = (np.arange(H * V, dtype=np.float32).reshape(H, V) % 17) - 8
    h = np.zeros((2, H), np.float32)
    h[0, 3] = 1.0
    h[1, 0] = 1.0
    cols = np.array([5, 0, 15, 5], np.int64)
    out = oracle.lmhead_logits(bf16(h), bf16(W), cols=cols)
    np.testing.assert_array_equal(out[0], W[3, cols])
    np.testing.assert_array_equal(out[1], W[0, cols])
