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
from gpu_helpers import (BF16_ATOL, BF16_RTOL, FP8_ATOL,
                         assert_attention_close, ensure_built,
                         oracle_attention, rows_of)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed, prefixes, q_len=8, kv_dtype="bf16", page_size=64):
    return wl.make_attention_inputs(
        batch=len(prefixes), q_len=q_len, num_q_heads=24, num_kv_heads=4,
        head_dim=256, page_size=page_size, prefix_lens=prefixes, seed=seed,
        device=DEV, kv_dtype=kv_dtype)


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_via_abi(inp, q_lens=None):
    """Call spec_verify_attention_noalloc through the C ABI."""
    lib = _native.load()
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"],
                       q_lens=q_lens)
    out = torch.full_like(inp["q"], float("nan"))
    rc = lib.spec_verify_attention_noalloc(
        ctypes.byref(desc), _vp(inp["q"]), _vp(inp["k_pages"]),
        _vp(inp["v_pages"]), _vp(inp["k_scales"]), _vp(inp["v_scales"]),
        _vp(inp["page_table"]), _vp(inp["seq_lens"]), inp["scale"],
        _vp(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.spec_last_error()
    return out


def _with_workspace(inp, q_lens=None):
    return sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                               inp["page_table"], inp["seq_lens"],
                               scale=inp["scale"], k_scales=inp["k_scales"],
                               v_scales=inp["v_scales"], q_lens=q_lens)


def _close(got, ref, fp8):
    g, r = got.float(), ref.float()
    assert torch.isfinite(g).all()
    bound = FP8_ATOL if fp8 else BF16_ATOL + BF16_RTOL * r.abs()
    assert torch.all((g - r).abs() <= bound)


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


def test_noalloc_ignores_what_an_earlier_call_left_in_the_scratch():
    ensure_built()
    # a larger call with NaN queries fills more partial slots with NaN than
    # the next call uses; the next call must read only what it wrote
    junk = _inputs(41, [30000, 25000, 20000, 9000], 16)
    junk["q"].fill_(float("nan"))
    _noalloc_via_abi(junk)
    inp = _inputs(42, [6000, 300, 11000])
    got = _noalloc_via_abi(inp)
    ref = _with_workspace(inp)
    torch.cuda.synchronize()
    _close(got, ref, False)
    assert_attention_close(rows_of(got), oracle_attention(inp), False,
                           "no-alloc after a NaN call")


@pytest.mark.parametrize("ps", [16, 64])
def test_noalloc_fp8_matches_workspace_entry_and_oracle(ps):
    ensure_built()
    inp = _inputs(50 + ps, [4000, 900, 7000], 8, kv_dtype="fp8_e4m3",
                  page_size=ps)
    for _ in range(2):  # two calls in a row
        got = _noalloc_via_abi(inp)
        ref = _with_workspace(inp)
        torch.cuda.synchronize()
        _close(got, ref, True)
    assert_attention_close(rows_of(got), oracle_attention(inp), True,
                           f"no-alloc FP8 page_size={ps}")


def test_noalloc_ragged_widths_match_workspace_entry_and_oracle():
    ensure_built()
    import oracle
    inp = _inputs(61, [3000, 64, 9000, 5], 16)
    ql = torch.tensor([16, 3, 9, 0], dtype=torch.int32, device=DEV)
    got = _noalloc_via_abi(inp, q_lens=ql)
    ref = _with_workspace(inp, q_lens=ql)
    torch.cuda.synchronize()
    _close(got, ref, False)
    bits = wl.to_numpy_bits
    exp = oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        num_kv_heads=4, scale=inp["scale"], q_lens=ql.cpu().numpy())
    assert_attention_close(rows_of(got), exp, False, "no-alloc ragged")


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
