"""ctypes binding of libspecverify (argument marshalling only).

Every step of the verify path runs in the CUDA library; this module turns torch
tensors into device pointers, allocates outputs and the workspace with torch
when the caller does not pass them, and raises on a non-OK status.  There is
no CPU fallback: if the library is missing or fails to load, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SV_OK = 0
SV_F32, SV_BF16 = 0, 1
SV_MODE_SAMPLE, SV_MODE_GREEDY, SV_MODE_LMHEAD, SV_MODE_DRAFT = 0, 1, 2, 3
FLAG_ZERO_MASS, FLAG_NONFINITE, FLAG_RESIDUAL_FALLBACK, FLAG_TIMEOUT, FLAG_BAD_TOKEN = 1, 2, 4, 8, 16

EXPORTS = ("sv_workspace_bytes", "sv_workspace_init", "spec_verify", "spec_verify_opts",
           "spec_verify_greedy", "spec_lmhead_verify", "spec_lmhead_draft",
           "spec_lmhead_verify_drafted",
           "sv_set_timing_events", "sv_test_lmhead_stall", "sv_status_string", "sv_version")


class Options(ctypes.Structure):
    """sv_options of include/specverify.h."""
    _fields_ = [("lenience", ctypes.c_float), ("top_k", ctypes.c_int32),
                ("top_p", ctypes.c_float), ("sampler", ctypes.c_int32)]


SV_SAMPLER_GUMBEL, SV_SAMPLER_INVERSE = 0, 1
SAMPLERS = {"gumbel": SV_SAMPLER_GUMBEL, "inverse": SV_SAMPLER_INVERSE}


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what} failed: {status_string(status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the in-tree libspecverify.so (building it with nvcc if absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"libspecverify is not built ({path}); run __graft_entry__.build()")
            _build.build()
        L = ctypes.CDLL(path)
        P, I, I64, U64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                  ctypes.c_float, ctypes.c_size_t)
        L.sv_workspace_bytes.argtypes = [I, I, I64, I]
        L.sv_workspace_bytes.restype = SZ
        L.sv_workspace_init.argtypes = [P, SZ, P]
        L.sv_workspace_init.restype = I
        L.spec_verify.argtypes = [P, P, P, I, I, I64, I, F, P, U64, U64, P, P, P, P, P, P, P, SZ, P]
        L.spec_verify.restype = I
        L.spec_verify_opts.argtypes = [P, P, P, I, I, I64, I, F, P, U64, U64, P, P, P, P, P, P,
                                       P, P, SZ, P]
        L.spec_verify_opts.restype = I
        L.spec_verify_greedy.argtypes = [P, P, I, I, I64, I, P, P, P, SZ, P]
        L.spec_verify_greedy.restype = I
        L.spec_lmhead_verify.argtypes = [P, P, I, P, P, I, P, I, I, I64, F, U64, U64, P, P, P, P,
                                         P, P, P, SZ, P]
        L.spec_lmhead_verify.restype = I
        L.spec_lmhead_draft.argtypes = [P, P, I, I, I64, F, U64, U64, I, P, P, P, P, P, P, SZ, P]
        L.spec_lmhead_verify_drafted.argtypes = [P, P, I, P, P, I, P, P, P, I, I, I64, F, U64,
                                                 U64, P, P, P, P, P, P, P, SZ, P]
        L.spec_lmhead_verify_drafted.restype = I
        L.spec_lmhead_draft.restype = I
        L.sv_set_timing_events.argtypes = [P, I]
        L.sv_set_timing_events.restype = I
        L.sv_test_lmhead_stall.argtypes = [I, ctypes.c_uint32]
        L.sv_test_lmhead_stall.restype = I
        L.sv_status_string.argtypes = [I]
        L.sv_status_string.restype = ctypes.c_char_p
        L.sv_version.argtypes = []
        L.sv_version.restype = I
        _lib = L
        return _lib


def test_lmhead_stall(job: int, wait_limit: int = 0) -> None:
    """Test only: the next fused LM-head calls withhold one accumulator hand-over
    (job < 0: none) and give up every bounded wait after `wait_limit` tries (0: the
    default); see sv_test_lmhead_stall in include/specverify.h."""
    load().sv_test_lmhead_stall(int(job), int(wait_limit))


def status_string(status: int) -> str:
    return load().sv_status_string(int(status)).decode()


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the library has no CPU path)")
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


class _WorkspaceCache:
    """Workspaces, one per (device, stream), grown on demand.  Calls queued on
    one stream may share a workspace; the library needs no initial contents."""

    def __init__(self):
        self._bufs = {}

    def get(self, nbytes: int, device, stream_key):
        torch = _torch()
        key = (str(device), stream_key)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf


_ws_cache = _WorkspaceCache()


def workspace_bytes(B: int, gamma: int, V: int, mode: int) -> int:
    return int(load().sv_workspace_bytes(int(B), int(gamma), int(V), int(mode)))


def alloc_workspace(B: int, gamma: int, V: int, mode: int, device="cuda"):
    torch = _torch()
    return torch.zeros(max(workspace_bytes(B, gamma, V, mode), 256), dtype=torch.uint8,
                       device=device)


def spec_verify(target_logits, draft_logits, draft_tokens, *, temperature: float = 1.0,
                row_temperature=None, seed: int = 0, round: int = 0, want_pq: bool = True,
                want_alpha: bool = False, want_flags: bool = True, out=None, workspace=None,
                stream=None, lenience: float = 1.0, top_k: int = 0, top_p: float = 1.0,
                sampler: str = "gumbel"):
    """Sampling verify through the C ABI.  Returns a dict of device tensors:
    tokens [B, g+1] int32, counts [B] int32, p/q [B, g] float32 (if want_pq),
    alpha [B] float32 (if want_alpha), flags [B] uint8 (if want_flags).
    lenience: l in (0, 1] (spec_verify_opts; 1 = the exact round).
    top_k: adjust every row to its k largest logits, ties kept (0 = off).
    top_p: then to its nucleus of probability top_p (1 = off).
    sampler: "gumbel" (the round's contract) or "inverse" (the opt-in inverse
    transform) for the target's own token."""
    torch = _torch()
    L = load()
    B, g1, V = target_logits.shape
    g = g1 - 1
    if tuple(draft_logits.shape) != (B, g, V) or tuple(draft_tokens.shape) != (B, g):
        raise ValueError("shape mismatch: target [B,g+1,V], draft [B,g,V], tokens [B,g]")
    if draft_logits.dtype != target_logits.dtype or draft_tokens.dtype != torch.int32:
        raise TypeError("draft logits must match target dtype; draft tokens must be int32")
    _check_cuda(target_logits, draft_logits, draft_tokens, row_temperature)
    dev = target_logits.device
    o = dict(out or {})
    if "tokens" not in o:
        o["tokens"] = torch.empty((B, g1), dtype=torch.int32, device=dev)
    if "counts" not in o:
        o["counts"] = torch.empty((B,), dtype=torch.int32, device=dev)
    if want_pq:
        o.setdefault("p", torch.empty((B, g), dtype=torch.float32, device=dev))
        o.setdefault("q", torch.empty((B, g), dtype=torch.float32, device=dev))
    if want_alpha:
        o.setdefault("alpha", torch.empty((B,), dtype=torch.float32, device=dev))
    if want_flags:
        o.setdefault("flags", torch.empty((B,), dtype=torch.uint8, device=dev))
    sh = _stream_handle(stream)
    need = workspace_bytes(B, g, V, SV_MODE_SAMPLE)
    ws = workspace if workspace is not None else _ws_cache.get(need, dev, sh.value)
    opts = Options(float(lenience), int(top_k), float(top_p), SAMPLERS[sampler])
    rc = L.spec_verify_opts(_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, g,
                            V, _dtype_code(target_logits), float(temperature),
                            _ptr(row_temperature), int(seed) & (2**64 - 1),
                            int(round) & (2**64 - 1), _ptr(o["tokens"]), _ptr(o["counts"]),
                            _ptr(o.get("p")), _ptr(o.get("q")), _ptr(o.get("alpha")),
                            _ptr(o.get("flags")), ctypes.addressof(opts), _ptr(ws), ws.numel(),
                            sh)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify")
    return o


def spec_verify_greedy(target_logits, draft_tokens, *, out=None, workspace=None, stream=None):
    """Greedy verify through the C ABI.  Returns tokens [B, g+1], counts [B]."""
    torch = _torch()
    L = load()
    B, g1, V = target_logits.shape
    g = g1 - 1
    if tuple(draft_tokens.shape) != (B, g) or draft_tokens.dtype != torch.int32:
        raise ValueError("draft tokens must be int32 [B, gamma]")
    _check_cuda(target_logits, draft_tokens)
    dev = target_logits.device
    o = dict(out or {})
    o.setdefault("tokens", torch.empty((B, g1), dtype=torch.int32, device=dev))
    o.setdefault("counts", torch.empty((B,), dtype=torch.int32, device=dev))
    sh = _stream_handle(stream)
    need = workspace_bytes(B, g, V, SV_MODE_GREEDY)
    ws = workspace if workspace is not None else _ws_cache.get(need, dev, sh.value)
    rc = L.spec_verify_greedy(_ptr(target_logits), _ptr(draft_tokens), B, g, V,
                              _dtype_code(target_logits), _ptr(o["tokens"]), _ptr(o["counts"]),
                              _ptr(ws), ws.numel(), sh)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_greedy")
    return o


def spec_lmhead_verify(h_target, W_target, h_draft, W_draft, draft_tokens, *, B: int,
                       gamma: int, temperature: float = 1.0, seed: int = 0, round: int = 0,
                       want_pq: bool = True, want_flags: bool = True, debug_logits=None,
                       out=None, workspace=None, stream=None):
    """Fused LM heads + sampling verify through the C ABI (bf16 inputs)."""
    torch = _torch()
    L = load()
    Mt, Ht = h_target.shape
    Md, Hd = h_draft.shape
    V = W_target.shape[1]
    if Mt != B * (gamma + 1) or Md != B * gamma or tuple(W_target.shape) != (Ht, V) or \
            tuple(W_draft.shape) != (Hd, V) or tuple(draft_tokens.shape) != (B, gamma):
        raise ValueError("shape mismatch in spec_lmhead_verify")
    _check_cuda(h_target, W_target, h_draft, W_draft, draft_tokens, debug_logits)
    dev = h_target.device
    o = dict(out or {})
    o.setdefault("tokens", torch.empty((B, gamma + 1), dtype=torch.int32, device=dev))
    o.setdefault("counts", torch.empty((B,), dtype=torch.int32, device=dev))
    if want_pq:
        o.setdefault("p", torch.empty((B, gamma), dtype=torch.float32, device=dev))
        o.setdefault("q", torch.empty((B, gamma), dtype=torch.float32, device=dev))
    if want_flags:
        o.setdefault("flags", torch.empty((B,), dtype=torch.uint8, device=dev))
    sh = _stream_handle(stream)
    need = workspace_bytes(B, gamma, V, SV_MODE_LMHEAD)
    ws = workspace if workspace is not None else _ws_cache.get(need, dev, sh.value)
    rc = L.spec_lmhead_verify(_ptr(h_target), _ptr(W_target), Ht, _ptr(h_draft), _ptr(W_draft),
                              Hd, _ptr(draft_tokens), B, gamma, V, float(temperature),
                              int(seed) & (2**64 - 1), int(round) & (2**64 - 1),
                              _ptr(o["tokens"]), _ptr(o["counts"]), _ptr(o.get("p")),
                              _ptr(o.get("q")), _ptr(o.get("flags")), _ptr(debug_logits),
                              _ptr(ws), ws.numel(), sh)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_lmhead_verify")
    return o


def spec_lmhead_verify_drafted(h_target, W_target, h_draft, W_draft, draft_tokens, draft_lse,
                               draft_logit, *, B: int, gamma: int, temperature: float = 1.0,
                               seed: int = 0, round: int = 0, want_pq: bool = True,
                               want_flags: bool = True, debug_logits=None, out=None,
                               workspace=None, stream=None):
    """spec_lmhead_verify with the draft rows' statistics from the draft step
    (draft_lse, draft_logit [B, gamma] float32, spec_lmhead_draft's lse and logit)."""
    torch = _torch()
    L = load()
    Mt, Ht = h_target.shape
    Md, Hd = h_draft.shape
    V = W_target.shape[1]
    if Mt != B * (gamma + 1) or Md != B * gamma or tuple(W_target.shape) != (Ht, V) or \
            tuple(W_draft.shape) != (Hd, V) or tuple(draft_tokens.shape) != (B, gamma) or \
            tuple(draft_lse.shape) != (B, gamma) or tuple(draft_logit.shape) != (B, gamma):
        raise ValueError("shape mismatch in spec_lmhead_verify_drafted")
    _check_cuda(h_target, W_target, h_draft, W_draft, draft_tokens, draft_lse, draft_logit,
                debug_logits)
    dev = h_target.device
    o = dict(out or {})
    o.setdefault("tokens", torch.empty((B, gamma + 1), dtype=torch.int32, device=dev))
    o.setdefault("counts", torch.empty((B,), dtype=torch.int32, device=dev))
    if want_pq:
        o.setdefault("p", torch.empty((B, gamma), dtype=torch.float32, device=dev))
        o.setdefault("q", torch.empty((B, gamma), dtype=torch.float32, device=dev))
    if want_flags:
        o.setdefault("flags", torch.empty((B,), dtype=torch.uint8, device=dev))
    sh = _stream_handle(stream)
    need = workspace_bytes(B, gamma, V, SV_MODE_LMHEAD)
    ws = workspace if workspace is not None else _ws_cache.get(need, dev, sh.value)
    rc = L.spec_lmhead_verify_drafted(
        _ptr(h_target), _ptr(W_target), Ht, _ptr(h_draft), _ptr(W_draft), Hd,
        _ptr(draft_tokens), _ptr(draft_lse), _ptr(draft_logit), B, gamma, V,
        float(temperature), int(seed) & (2**64 - 1), int(round) & (2**64 - 1),
        _ptr(o["tokens"]), _ptr(o["counts"]), _ptr(o.get("p")), _ptr(o.get("q")),
        _ptr(o.get("flags")), _ptr(debug_logits), _ptr(ws), ws.numel(), sh)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_lmhead_verify_drafted")
    return o


def spec_lmhead_draft(h_draft, W_draft, *, pos: int, temperature: float = 1.0, seed: int = 0,
                      round: int = 0, debug_logits=None, out=None, workspace=None,
                      stream=None):
    """Draft LM head + draw of one draft position through the C ABI (bf16 inputs).
    Returns tokens [B] int32, q [B] float32 (q(x)), lse [B] float32, logit [B] float32."""
    torch = _torch()
    L = load()
    B, Hd = h_draft.shape
    V = W_draft.shape[1]
    if tuple(W_draft.shape) != (Hd, V):
        raise ValueError("shape mismatch in spec_lmhead_draft")
    _check_cuda(h_draft, W_draft, debug_logits)
    dev = h_draft.device
    o = dict(out or {})
    o.setdefault("tokens", torch.empty((B,), dtype=torch.int32, device=dev))
    o.setdefault("q", torch.empty((B,), dtype=torch.float32, device=dev))
    o.setdefault("lse", torch.empty((B,), dtype=torch.float32, device=dev))
    o.setdefault("logit", torch.empty((B,), dtype=torch.float32, device=dev))
    sh = _stream_handle(stream)
    need = workspace_bytes(B, 1, V, SV_MODE_DRAFT)
    ws = workspace if workspace is not None else _ws_cache.get(need, dev, sh.value)
    rc = L.spec_lmhead_draft(_ptr(h_draft), _ptr(W_draft), Hd, B, V, float(temperature),
                             int(seed) & (2**64 - 1), int(round) & (2**64 - 1), int(pos),
                             _ptr(o["tokens"]), _ptr(o["q"]), _ptr(o["lse"]), _ptr(o["logit"]),
                             _ptr(debug_logits), _ptr(ws), ws.numel(), sh)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_lmhead_draft")
    return o
