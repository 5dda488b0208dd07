"""libspecverify: the verify-and-sample step of speculative decoding on GB300.

The product is the C-ABI shared library built from ``csrc/`` (see
``include/specverify.h``); this package holds its build script, a thin ctypes
binding with the same entry-point names, and the seeded synthetic workloads
used by the tests and the benchmark.
"""
from ._lib import (FLAG_BAD_TOKEN, FLAG_NONFINITE, FLAG_RESIDUAL_FALLBACK, FLAG_TIMEOUT,
                   FLAG_ZERO_MASS, SpecVerifyError, alloc_workspace, library_path, load,
                   spec_lmhead_draft, spec_lmhead_verify, spec_lmhead_verify_drafted,
                   spec_verify, spec_verify_greedy, status_string, test_lmhead_stall,
                   workspace_bytes)

__all__ = ["spec_verify", "spec_verify_greedy", "spec_lmhead_verify", "spec_lmhead_draft",
           "spec_lmhead_verify_drafted",
           "workspace_bytes",
           "alloc_workspace", "load", "library_path", "status_string", "SpecVerifyError",
           "FLAG_ZERO_MASS", "FLAG_NONFINITE", "FLAG_RESIDUAL_FALLBACK", "FLAG_TIMEOUT",
           "FLAG_BAD_TOKEN", "test_lmhead_stall"]
