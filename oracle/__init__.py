"""CPU oracle for the speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` leg of ``bench.py`` import this
package.  The product path (the CUDA library and its Python binding) never
imports it and shares no source with it.

The arithmetic lives in ``sv_oracle.c`` (plain single-threaded C, double
precision); this module builds it with gcc on first use and wraps it with
ctypes + numpy.  ``exact.py`` (exact rational enumeration) and
``theory.py`` (the pages' closed forms) complete the oracle.

Functions whose outputs are pinned (see ``tests/test_oracle_*.py``): Philox
(statistics here, cuRAND on a GPU), the accept/residual arithmetic (worked
examples of three pages), the full verify (chi-square, 1-TV, equation (1),
tokens-per-run histogram, exhaustive enumeration, the T->0 limit), greedy
(brute force), the LM-head logits (float64 matmul of the same bf16 values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_HDR = os.path.join(_HERE, "sv_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

F32, BF16 = 0, 1
FLAG_ZERO_MASS, FLAG_NONFINITE, FLAG_RESIDUAL_FALLBACK, FLAG_BAD_TOKEN = 1, 2, 4, 16

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no machine-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_SO)) or any(
        os.path.getmtime(p) > os.path.getmtime(_SO) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            L.svo_philox4x32_10.argtypes = [P, P, P]
            L.svo_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                      ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint32,
                                      ctypes.c_int]
            L.svo_uniform.restype = ctypes.c_double
            L.svo_uniform_row.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64,
                                          ctypes.c_int64, P]
            L.svo_draw_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                           ctypes.c_uint64]
            L.svo_draw_uniform.restype = ctypes.c_double
            for name in ("svo_accept_mass", "svo_residual"):
                getattr(L, name).argtypes = [P, P, ctypes.c_int64, P]
                getattr(L, name).restype = ctypes.c_double
            L.svo_softmax.argtypes = [P, ctypes.c_int64, P]
            L.svo_softmax.restype = ctypes.c_double
            L.svo_spec_verify.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_float, P, ctypes.c_uint64,
                                          ctypes.c_uint64, P, P, P, P, P, P, P, P, P, P]
            L.svo_spec_verify.restype = ctypes.c_int
            L.svo_spec_verify_rows.argtypes = L.svo_spec_verify.argtypes + [ctypes.c_int,
                                                                            ctypes.c_int]
            L.svo_spec_verify_rows.restype = ctypes.c_int
            L.svo_spec_verify_ex.argtypes = L.svo_spec_verify_rows.argtypes + [P]
            L.svo_spec_verify_ex.restype = ctypes.c_int
            L.svo_spec_verify_greedy.argtypes = [P, P, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int64, ctypes.c_int, P, P]
            L.svo_spec_verify_greedy.restype = ctypes.c_int
            L.svo_draft_sample.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                           ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int, P, P,
                                           P, P]
            L.svo_draft_sample.restype = ctypes.c_int
            L.svo_lmhead_logits.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                            P, ctypes.c_int64, P]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().svo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed, tag, pos, b, rnd, c0, lane) -> float:
    return lib().svo_uniform(seed, tag, pos, b, rnd, c0, lane)


def draw_uniform(seed, pos, b, rnd) -> float:
    """The uniform U in [0, 1) (53 bits) of the inverse-transform draw at position pos."""
    return lib().svo_draw_uniform(int(seed) & (2**64 - 1), pos, b, int(rnd) & (2**64 - 1))


def uniform_row(seed, tag, pos, b, rnd, v0, n) -> np.ndarray:
    out = np.zeros(int(n), np.float64)
    lib().svo_uniform_row(seed, tag, pos, b, rnd, v0, n, _ptr(out))
    return out


def accept_mass(p, q):
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.zeros_like(p)
    beta = lib().svo_accept_mass(_ptr(p), _ptr(q), p.size, _ptr(out))
    return beta, out


def residual(p, q):
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.zeros_like(p)
    mass = lib().svo_residual(_ptr(p), _ptr(q), p.size, _ptr(out))
    return mass, out


def softmax(s):
    s = np.ascontiguousarray(s, dtype=np.float64)
    out = np.zeros_like(s)
    S = lib().svo_softmax(_ptr(s), s.size, _ptr(out))
    return S, out


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # raw bf16 bit patterns
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


class _Options(ctypes.Structure):
    """svo_options (sv_oracle.h)."""
    _fields_ = [("lenience", ctypes.c_double), ("top_k", ctypes.c_int),
                ("top_p", ctypes.c_double), ("nucleus_gap", ctypes.c_void_p),
                ("sampler", ctypes.c_int)]


SAMPLERS = {"gumbel": 0, "inverse": 1}


def spec_verify(zt, zd, xt, temperature=1.0, row_temperature=None, seed=0, rnd=0,
                want_beta=False, rows=None, threads=1, lenience=1.0, top_k=0, top_p=1.0,
                sampler="gumbel"):
    """Sampling verify.  zt [B,g+1,V], zd [B,g,V] (float32 or bf16 bits as uint16),
    xt [B,g] int32.  Returns a dict of numpy arrays.

    lenience: l in (0, 1]; a draft is accepted iff u <= p / (l q) (1: exact).
    top_k: keep the entries of every row at or above its k-th largest logit (0: off).
    top_p: then keep each row's nucleus of probability top_p (1: off); the output
    "nucleus_gap" [B] is the smallest distance of top_p from a cut's cumulative
    probabilities in the batch row.

    sampler: how the target's own token (residual or bonus) is drawn.  "gumbel"
    (default): argmax of log w_v + g_v with Gumbel noise from Philox tag 1 at the
    draw position, ties to the lowest index; "gap" [B] is the top-1 minus top-2
    key (natural-log units; inf with one candidate, NaN for an empty row).
    "inverse": the inverse transform with one 53-bit uniform U; "gap" [B] is the
    distance of U W from the nearer end of the drawn token's cumulative interval
    (probability units).

    rows: optional list of batch-row indices to compute (others left zero);
    threads: run disjoint row ranges in that many Python threads (each a plain
    single-threaded oracle call; ctypes releases the GIL)."""
    zt = np.ascontiguousarray(zt)
    zd = np.ascontiguousarray(zd)
    xt = np.ascontiguousarray(xt, dtype=np.int32)
    B, g1, V = zt.shape
    g = g1 - 1
    assert zd.shape == (B, g, V) and xt.shape == (B, g) and zd.dtype == zt.dtype
    rowT = None if row_temperature is None else np.ascontiguousarray(row_temperature, np.float32)
    out = dict(
        tokens=np.zeros((B, g + 1), np.int32), counts=np.zeros(B, np.int32),
        p=np.zeros((B, g)), q=np.zeros((B, g)), ratio=np.zeros((B, g)), u=np.zeros((B, g)),
        beta=np.zeros((B, g)) if want_beta else None, gap=np.zeros(B), resid_mass=np.zeros(B),
        flags=np.zeros(B, np.uint8))
    L = lib()

    out["nucleus_gap"] = np.full(B, np.inf)
    opt = _Options(float(lenience), int(top_k), float(top_p), _ptr(out["nucleus_gap"]),
                   SAMPLERS[sampler])

    def run(b0, b1):
        rc = L.svo_spec_verify_ex(
            _ptr(zt), _ptr(zd), _ptr(xt), B, g, V, _dtype_code(zt), float(temperature),
            _ptr(rowT), int(seed) & (2**64 - 1), int(rnd) & (2**64 - 1), _ptr(out["tokens"]),
            _ptr(out["counts"]), _ptr(out["p"]), _ptr(out["q"]), _ptr(out["ratio"]),
            _ptr(out["u"]), _ptr(out["beta"]), _ptr(out["gap"]), _ptr(out["resid_mass"]),
            _ptr(out["flags"]), int(b0), int(b1), ctypes.byref(opt))
        if rc != 0:
            raise ValueError(f"oracle spec_verify rejected its arguments (rc={rc})")

    ranges = [(b, b + 1) for b in rows] if rows is not None else [(0, B)]
    if threads > 1 and rows is None and B > 1:
        step = -(-B // threads)
        ranges = [(b, min(B, b + step)) for b in range(0, B, step)]
    if threads > 1 and len(ranges) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda r: run(*r), ranges))
    else:
        for r in ranges:
            run(*r)
    if want_beta:
        out["alpha"] = out["beta"].mean(axis=1)
    return out


def spec_verify_greedy(zt, xt):
    zt = np.ascontiguousarray(zt)
    xt = np.ascontiguousarray(xt, dtype=np.int32)
    B, g1, V = zt.shape
    g = g1 - 1
    assert xt.shape == (B, g)
    tokens = np.zeros((B, g + 1), np.int32)
    counts = np.zeros(B, np.int32)
    rc = lib().svo_spec_verify_greedy(_ptr(zt), _ptr(xt), B, g, V, _dtype_code(zt),
                                      _ptr(tokens), _ptr(counts))
    if rc != 0:
        raise ValueError(f"oracle spec_verify_greedy rejected its arguments (rc={rc})")
    return dict(tokens=tokens, counts=counts)


def draft_sample(logits, temperature=1.0, seed=0, rnd=0, pos=0):
    """Draft sampling of one position from logits [B, V] (float32): Gumbel-max with
    Philox tag 2.  Returns tokens [B], q [B] = q(x), lse [B], gap [B]."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    B, V = z.shape
    out = dict(tokens=np.zeros(B, np.int32), q=np.zeros(B), lse=np.zeros(B), gap=np.zeros(B))
    rc = lib().svo_draft_sample(_ptr(z), B, V, float(temperature), int(seed) & (2**64 - 1),
                                int(rnd) & (2**64 - 1), int(pos), _ptr(out["tokens"]),
                                _ptr(out["q"]), _ptr(out["lse"]), _ptr(out["gap"]))
    if rc != 0:
        raise ValueError(f"oracle draft_sample rejected its arguments (rc={rc})")
    return out


def lmhead_logits(h_bits, W_bits, cols=None):
    """logits[M, ncols] = h W[:, cols] in float64, from bf16 bit patterns (uint16)."""
    h = np.ascontiguousarray(h_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    M, H = h.shape
    H2, V = W.shape
    assert H == H2
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nc = V if c is None else c.size
    out = np.zeros((M, nc), np.float32)
    lib().svo_lmhead_logits(_ptr(h), _ptr(W), M, H, V, _ptr(c), nc, _ptr(out))
    return out
