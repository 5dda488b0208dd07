"""Failure detection of the fused LM head without a GPU fault.

The bounded waits of the GEMM pass are made to run out on purpose: through the
test-only sv_test_lmhead_stall, the first CTA never hands one accumulator to
its epilogue, so the epilogue's wait on it gives up after a short limit.  The
CTA then ends its other roles, lets its copies land, frees its tensor memory
and returns; the call returns normally with every batch row flagged
SV_FLAG_TIMEOUT, and the next call on the same context gives the results of a
call that never stalled.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_21_gb300 as sv
from tests._parity import to_np
from tests.test_gpu_lmhead import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load()


def _call(case, B, gamma):
    h_t, W_t, h_d, W_d, xt = case
    o = sv.spec_lmhead_verify(h_t, W_t, h_d, W_d, xt, B=B, gamma=gamma, seed=3, round=1)
    torch.cuda.synchronize()
    return to_np(o)


def test_stalled_hand_over_times_out_and_the_context_survives():
    B, gamma = 4, 2
    case = make_case(B, gamma, 4096, 256, 256, seed=5)
    ref = _call(case, B, gamma)
    assert not np.any(ref["flags"] & sv.FLAG_TIMEOUT)
    sv.test_lmhead_stall(0, 1 << 12)
    try:
        stalled = _call(case, B, gamma)
    finally:
        sv.test_lmhead_stall(-1, 0)
    assert np.all(stalled["flags"] & sv.FLAG_TIMEOUT), stalled["flags"]
    assert stalled["tokens"].min() >= -1 and stalled["tokens"].max() < 4096
    again = _call(case, B, gamma)
    for k in ("tokens", "counts", "p", "q", "flags"):
        np.testing.assert_array_equal(again[k], ref[k], err_msg=k)
