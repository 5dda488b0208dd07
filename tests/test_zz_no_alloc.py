"""spec_verify_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (a plugin handed only its input and output buffers, code that must
not enter an allocator on the hot path) get the sampling verify with its scratch
memory in a static 4 MiB device array inside the library.  This test calls it
through the C ABI and checks its outputs against spec_verify's (which uses a
caller-supplied workspace) on two calls in a row, with the tolerance the other
parity tests use.  It lives in its own file, collected last, so that a run that
stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_21_gb300 as sv
from speculative_decoding_verification_21_gb300 import workloads as wl

REL_TOL = 1e-5
LIMIT = 4 << 20


def _noalloc_fn():
    L = sv.load()
    P, I, I64, U64, F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                         ctypes.c_float)
    fn = L.spec_verify_noalloc
    fn.argtypes = [P, P, P, I, I, I64, I, F, P, U64, U64, P, P, P, P, P, P, P]
    fn.restype = I
    return fn


def _call_noalloc(w, seed, rnd, stream):
    fn = _noalloc_fn()
    B, g = w.B, w.gamma
    dev = w.zt.device
    out = dict(tokens=torch.full((B, g + 1), -7, dtype=torch.int32, device=dev),
               counts=torch.full((B,), -7, dtype=torch.int32, device=dev),
               p=torch.full((B, g), -1.0, device=dev), q=torch.full((B, g), -1.0, device=dev),
               alpha=torch.full((B,), -1.0, device=dev),
               flags=torch.full((B,), 255, dtype=torch.uint8, device=dev))
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = fn(P(w.zt), P(w.zd), P(w.xt), B, g, w.V, 1 if w.zt.dtype == torch.bfloat16 else 0,
            w.temperature, P(w.row_temperature), seed, rnd, P(out["tokens"]), P(out["counts"]),
            P(out["p"]), P(out["q"]), P(out["alpha"]), P(out["flags"]),
            ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, sv.status_string(rc)
    return out


def _close(a, b):
    a, b = a.cpu().numpy().astype(np.float64), b.cpu().numpy().astype(np.float64)
    return np.all(np.abs(a - b) <= REL_TOL * np.abs(b) + 1e-37)


@pytest.mark.gpu
def test_noalloc_matches_spec_verify_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    # two calls in a row with different sizes, so the second starts from the
    # first call's leftovers in the shared scratch array
    # a third case in fp32 logits with a per-row temperature
    w3 = wl.sample_b64(sigma=1.0, B=16, gamma=2, V=4000, seed=79)
    w3.zt, w3.zd = w3.zt.float().contiguous(), w3.zd.float().contiguous()
    w3.row_temperature = torch.linspace(0.5, 1.5, w3.B, device=w3.zt.device)
    cases = [(wl.sample_b64(sigma=1.0, B=32, gamma=4, V=50000, seed=77), 5, 0),
             (wl.sample_b64(sigma=0.5, B=48, gamma=3, V=32771, seed=78), 5, 1),
             (w3, 6, 2)]
    for w, seed, rnd in cases:
        assert sv.workspace_bytes(w.B, w.gamma, w.V, 0) <= LIMIT
        got = _call_noalloc(w, seed, rnd, stream)
        ref = sv.spec_verify(w.zt, w.zd, w.xt, temperature=w.temperature,
                             row_temperature=w.row_temperature, seed=seed, round=rnd,
                             want_alpha=True)
        torch.cuda.synchronize()
        assert torch.equal(got["tokens"], ref["tokens"])
        assert torch.equal(got["counts"], ref["counts"])
        assert torch.equal(got["flags"], ref["flags"])
        for k in ("p", "q", "alpha"):
            assert _close(got[k], ref[k]), k


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # validated before any device work: no GPU needed
    fn = _noalloc_fn()
    fake = ctypes.c_void_p(0x10000)
    B, g, V = 2048, 8, 152064
    assert sv.workspace_bytes(B, g, V, 0) > LIMIT
    rc = fn(fake, fake, fake, B, g, V, 1, 1.0, None, 0, 0, fake, fake, None, None, None, None,
            None)
    assert rc == -4, sv.status_string(rc)
