"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every entry point its header declares, size the
workspace, and reject bad arguments with the documented status before any
kernel is queued.  Pointer arguments here are fake non-null addresses: a
validating call returns before touching them.
"""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_21_gb300 as sv
from speculative_decoding_verification_21_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_library_exports_every_declared_symbol():
    L = sv.load()
    names = declared_functions()
    assert "spec_verify" in names and "spec_verify_greedy" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in specverify.h but not exported"
    assert set(_lib.EXPORTS) <= set(names)


def test_version_and_status_strings():
    L = sv.load()
    assert L.sv_version() >= 100
    for st in (0, -1, -2, -3, -4, -5, -6):
        assert sv.status_string(st).startswith("SV_")


def test_workspace_sizes():
    assert sv.workspace_bytes(0, 4, 1000, 0) == 0
    a = sv.workspace_bytes(64, 4, 128256, 0)
    b = sv.workspace_bytes(128, 4, 128256, 0)
    assert 0 < a < b and a % 256 == 0
    assert sv.workspace_bytes(64, 5, 32000, 1) > 0
    assert sv.workspace_bytes(1, 0, 10, 0) == 0       # gamma out of range
    assert sv.workspace_bytes(1, 33, 10, 0) == 0
    assert sv.workspace_bytes(1, 4, 0, 0) == 0
    assert sv.workspace_bytes(1, 4, 2**31, 0) == 0


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced
FAKE_MIS = ctypes.c_void_p(0x10008)  # 8-byte aligned only


def _sv(L, zt=FAKE, zd=FAKE, xt=FAKE, B=2, g=2, V=64, dt=0, T=1.0, rowT=None, tok=FAKE,
        cnt=FAKE, ws=FAKE, wsb=1 << 20):
    return L.spec_verify(zt, zd, xt, B, g, V, dt, T, rowT, 0, 0, tok, cnt, None, None, None,
                         None, ws, wsb, None)


def _svo(L, lenience=1.0, top_k=0, top_p=1.0, opts=True, **kw):
    o = _lib.Options(lenience, top_k, top_p)
    a = dict(zt=FAKE, zd=FAKE, xt=FAKE, B=2, g=2, V=64, dt=0, T=1.0, tok=FAKE, cnt=FAKE, ws=FAKE,
             wsb=1 << 20)
    a.update(kw)
    return L.spec_verify_opts(a["zt"], a["zd"], a["xt"], a["B"], a["g"], a["V"], a["dt"], a["T"],
                              None, 0, 0, a["tok"], a["cnt"], None, None, None, None,
                              ctypes.addressof(o) if opts else None, a["ws"], a["wsb"], None)


def test_spec_verify_opts_argument_errors():
    L = sv.load()
    for bad in (0.0, -0.25, 1.0000001, 2.0, float("nan"), float("inf")):
        assert _svo(L, lenience=bad) == -1, bad
    assert _svo(L, top_k=-1) == -1
    for bad in (0.0, -0.5, 1.5, float("nan")):
        assert _svo(L, top_p=bad) == -1, bad
    # the remaining arguments are checked as by spec_verify
    assert _svo(L, lenience=0.5, g=0) == -1
    assert _svo(L, lenience=0.5, dt=7) == -2
    assert _svo(L, lenience=0.5, zt=FAKE_MIS) == -3
    assert _svo(L, lenience=0.5, ws=None) == -4
    assert _svo(L, opts=False, ws=None) == -4
    assert _svo(L, lenience=0.5, B=0) == 0  # nothing to do
    # nucleus sums are exact for V <= 2^21 only; no workspace, so nothing can launch
    big = (1 << 21) + 8
    assert _svo(L, top_p=0.9, V=big, ws=None) == -6
    assert _svo(L, top_p=0.9, V=1 << 21, ws=None) == -4
    assert _svo(L, top_p=1.0, V=big, ws=None) == -4
    assert _svo(L, top_k=50, V=big, ws=None) == -4


def test_spec_verify_argument_errors():
    L = sv.load()
    assert _sv(L, g=0) == -1
    assert _sv(L, g=33) == -1
    assert _sv(L, V=0) == -1
    assert _sv(L, B=-1) == -1
    assert _sv(L, dt=7) == -2
    assert _sv(L, T=0.0) == -1
    assert _sv(L, T=-1.0) == -1
    assert _sv(L, T=float("nan")) == -1
    assert _sv(L, zt=None) == -1
    assert _sv(L, tok=None) == -1
    assert _sv(L, zt=FAKE_MIS) == -3
    assert _sv(L, zd=FAKE_MIS) == -3
    assert _sv(L, ws=None) == -4
    assert _sv(L, wsb=16) == -4
    assert _sv(L, ws=ctypes.c_void_p(0x10010)) == -3
    assert _sv(L, B=0) == 0  # no-op, nothing queued


def test_greedy_argument_errors():
    L = sv.load()
    g = lambda **k: L.spec_verify_greedy(k.get("zt", FAKE), FAKE, k.get("B", 2), k.get("g", 2),
                                         k.get("V", 64), k.get("dt", 1), FAKE, FAKE,
                                         k.get("ws", FAKE), k.get("wsb", 1 << 20), None)
    assert g(g=0) == -1
    assert g(dt=3) == -2
    assert g(zt=FAKE_MIS) == -3
    assert g(wsb=8) == -4
    assert g(B=0) == 0


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    zt = torch.zeros(1, 2, 8)
    zd = torch.zeros(1, 1, 8)
    xt = torch.zeros(1, 1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        sv.spec_verify(zt, zd, xt)


def _lm(L, ht=FAKE, Wt=FAKE, Ht=128, hd=FAKE, Wd=FAKE, Hd=128, xt=FAKE, B=2, g=2, V=1024,
        T=1.0, tok=FAKE, cnt=FAKE, dbg=None, ws=FAKE, wsb=1 << 26):
    return L.spec_lmhead_verify(ht, Wt, Ht, hd, Wd, Hd, xt, B, g, V, T, 0, 0, tok, cnt, None,
                                None, None, dbg, ws, wsb, None)


def test_lmhead_argument_errors():
    L = sv.load()
    assert _lm(L, g=0) == -1
    assert _lm(L, T=0.0) == -1
    assert _lm(L, ht=None) == -1
    assert _lm(L, Wd=None) == -1
    assert _lm(L, Ht=100) == -6            # hidden sizes must be multiples of 64
    assert _lm(L, Hd=32) == -6
    assert _lm(L, Ht=16384 + 64) == -6     # beyond the compact-row copies
    assert _lm(L, B=52, g=4) == -6         # B*(gamma+1) = 260 > 256 token rows
    assert _lm(L, V=1001) == -6            # W rows must be 16-byte multiples
    assert _lm(L, Wt=FAKE_MIS) == -3
    assert _lm(L, hd=FAKE_MIS) == -3
    assert _lm(L, dbg=FAKE_MIS) == -3
    assert _lm(L, wsb=1024) == -4
    assert _lm(L, ws=None) == -4
    assert _lm(L, ws=ctypes.c_void_p(0x10010)) == -3
    assert _lm(L, B=0) == 0


def test_lmhead_workspace_size():
    need = sv.workspace_bytes(32, 4, 128256, 2)
    # compact copies of up to B hidden rows per side at the largest hidden size
    assert need >= 2 * 32 * 16384 * 2
    assert need % 256 == 0
    assert sv.workspace_bytes(64, 4, 128256, 2) > need


def test_lmhead_draft_argument_errors():
    L = sv.load()

    def call(h=FAKE, W=FAKE, Hd=128, B=4, V=1024, T=1.0, pos=0, tok=FAKE, ws=FAKE, wsb=1 << 22):
        return L.spec_lmhead_draft(h, W, Hd, B, V, T, 0, 0, pos, tok, None, None, None, None, ws,
                                   wsb, None)
    assert call(B=0) == 0
    assert call(T=0.0) == -1
    assert call(T=float("nan")) == -1
    assert call(V=0) == -1
    assert call(h=None) == -1
    assert call(tok=None) == -1
    assert call(pos=-1) == -1
    assert call(pos=1 << 24) == -1
    assert call(Hd=100) == -6
    assert call(Hd=16384 + 64) == -6
    assert call(B=129) == -6
    assert call(V=1001) == -6
    assert call(h=FAKE_MIS) == -3
    assert call(ws=None) == -4
    assert call(wsb=16) == -4


def test_draft_workspace_size():
    a = sv.workspace_bytes(32, 1, 128256, 3)
    assert a > 0 and a % 256 == 0
    assert sv.workspace_bytes(64, 1, 128256, 3) > a


def test_lmhead_verify_drafted_argument_errors():
    L = sv.load()

    def call(lse=FAKE, logit=FAKE, B=4, g=2, V=1024, T=1.0, Ht=128, ws=FAKE, wsb=1 << 26):
        return L.spec_lmhead_verify_drafted(FAKE, FAKE, Ht, FAKE, FAKE, 128, FAKE, lse, logit, B,
                                            g, V, T, 0, 0, FAKE, FAKE, None, None, None, None,
                                            ws, wsb, None)
    assert call(B=0) == 0
    assert call(lse=None) == -1
    assert call(logit=None) == -1
    assert call(T=0.0) == -1
    assert call(g=0) == -1
    assert call(lse=ctypes.c_void_p(0x10002)) == -3
    assert call(Ht=100) == -6
    assert call(ws=None) == -4


def test_timing_events_argument_check():
    """A non-NULL event array needs n >= 1; NULL switches recording off.  No event
    is recorded here (no call follows while they are set)."""
    L = sv.load()
    arr = (ctypes.c_void_p * 1)(ctypes.c_void_p(0x10000))
    assert L.sv_set_timing_events(ctypes.cast(arr, ctypes.c_void_p), 0) == -1
    assert L.sv_set_timing_events(None, 0) == 0
