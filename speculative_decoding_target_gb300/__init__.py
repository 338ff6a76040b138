"""Target-verify step of speculative decoding on one GB300 (sm_103a).

The compute lives in ``libspecverify.so`` (hand-written CUDA behind a C ABI,
``include/spec_verify.h``); ``_native`` is its ctypes binding.  Import of
this package does not load the library; the first call does, and raises if
it is missing.
"""
from ._native import (SpecError, accept_workspace_size, alloc_workspace,
                      desc_for, greedy_accept, greedy_accept_into, kv_append,
                      load,
                      make_desc, verify_attention, verify_attention_into,
                      verify_status, verify_workspace_size)

__all__ = [
    "SpecError", "accept_workspace_size", "alloc_workspace", "desc_for",
    "greedy_accept", "greedy_accept_into", "kv_append", "load", "make_desc",
    "verify_attention", "verify_attention_into", "verify_status",
    "verify_workspace_size",
]
