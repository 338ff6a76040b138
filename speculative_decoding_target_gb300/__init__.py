"""Target-verify step of speculative decoding on one GB300 (sm_103a).

The compute lives in ``libspecverify.so`` (hand-written CUDA behind a C ABI,
``include/spec_verify.h``); ``_native`` is its ctypes binding.  Import of
this package does not load the library; the first call does, and raises if
it is missing.
"""
from ._native import (SpecError, accept_workspace_size, alloc_workspace,
                      desc_for, dflash2_select, dflash2_select_into, greedy_accept, greedy_accept_commit,
                      greedy_accept_commit_into, greedy_accept_into,
                      kv_append, load, make_desc, prepare_next_block,
                      prepare_next_block_into, set_wait_limit, stochastic_accept,
                      stochastic_accept_into, stochastic_workspace_size,
                      verify_attention,
                      verify_attention_into, verify_status,
                      verify_workspace_size, width_policy)

__all__ = [
    "SpecError", "accept_workspace_size", "alloc_workspace", "desc_for",
    "dflash2_select", "dflash2_select_into",
    "greedy_accept", "greedy_accept_commit", "greedy_accept_commit_into",
    "greedy_accept_into", "kv_append", "load", "make_desc",
    "prepare_next_block", "prepare_next_block_into", "set_wait_limit",
    "stochastic_accept",
    "stochastic_accept_into", "stochastic_workspace_size", "verify_attention",
    "verify_attention_into", "verify_status", "verify_workspace_size",
    "width_policy",
]
