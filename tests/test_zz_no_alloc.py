"""The no-alloc verify entry point (for callers that cannot allocate device
memory, e.g. code handed only an engine's input and output buffers) matches
the workspace entry point.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import _native
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import BF16_ATOL, BF16_RTOL, ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, prefixes, q_len=8):
    return wl.make_attention_inputs(
        batch=len(prefixes), q_len=q_len, num_q_heads=24, num_kv_heads=4,
        head_dim=256, page_size=64, prefix_lens=prefixes, seed=seed,
        device=DEV)


def _noalloc_via_abi(inp):
    """Call spec_verify_attention_noalloc through the C ABI."""
    lib = _native.load()
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"])
    out = torch.full_like(inp["q"], float("nan"))
    rc = lib.spec_verify_attention_noalloc(
        ctypes.byref(desc), ctypes.c_void_p(inp["q"].data_ptr()),
        ctypes.c_void_p(inp["k_pages"].data_ptr()),
        ctypes.c_void_p(inp["v_pages"].data_ptr()), None, None,
        ctypes.c_void_p(inp["page_table"].data_ptr()),
        ctypes.c_void_p(inp["seq_lens"].data_ptr()), inp["scale"],
        ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.spec_last_error()
    return out


def _with_workspace(inp):
    return sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                               inp["page_table"], inp["seq_lens"],
                               scale=inp["scale"])


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    ensure_built()
    # two calls in a row on different shapes and lengths: the second must
    # not see anything the first left in the shared scratch
    cases = [_inputs(31, [5000, 700, 12000]), _inputs(32, [2048, 9000], 16)]
    for inp in cases:
        got = _noalloc_via_abi(inp)
        ref = _with_workspace(inp)
        torch.cuda.synchronize()
        g, r = got.float(), ref.float()
        assert torch.isfinite(g).all()
        assert torch.all((g - r).abs() <= BF16_ATOL + BF16_RTOL * r.abs())


def test_noalloc_rejects_shapes_beyond_its_scratch():
    ensure_built()
    lib = _native.load()
    desc = _native.make_desc(batch=1000, q_len=16, num_q_heads=32,
                             num_kv_heads=4, head_dim=256, page_size=64,
                             num_pages=1000, max_pages_per_seq=8)
    assert sv.verify_workspace_size(desc) > _native.NOALLOC_SCRATCH_BYTES
    rc = lib.spec_verify_attention_noalloc(
        ctypes.byref(desc), None, None, None, None, None, None, None, 0.0625,
        None, None)
    assert rc == _native.SPEC_ERR_WORKSPACE
    assert b"no-alloc" in lib.spec_last_error()
