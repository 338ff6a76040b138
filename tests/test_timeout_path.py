"""The split kernels' timeout path, exercised on the GPU without a hang.

Every mbarrier wait of the split kernels is bounded.  With a short bound set
through the C ABI's test hook (checked calls only), the first waits run out:
the CTA records SPEC_STATUS_TIMEOUT, stops issuing loads, drains the loads
and MMAs it already issued with the normal bound, frees its tensor memory
and exits.  The call's output is invalid; the test checks the status word
and that the next call on the same stream and workspace, with the normal
bound, is correct against the oracle.
"""
import pytest
import torch

import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import _native
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import (assert_attention_close, ensure_built,
                         oracle_attention, rows_of)

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (KV dtype, q_len, page size): the bf16 tcgen05 kernel; FP8 blocks of at
# most 64 rows per KV head (K and V^T as tensor-memory operands); FP8 blocks
# of more rows (the tcgen05 kernel's FP8 instance).
CASES = [("bf16", 8, 64), ("fp8_e4m3", 8, 64), ("fp8_e4m3", 16, 16)]


def _call(inp, ws):
    return sv.verify_attention(
        inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
        inp["seq_lens"], scale=inp["scale"], k_scales=inp["k_scales"],
        v_scales=inp["v_scales"], checked=True, workspace=ws)


@pytest.mark.parametrize("kv_dtype,q_len,ps", CASES)
def test_short_wait_bound_reports_timeout_and_the_next_call_is_correct(
        kv_dtype, q_len, ps):
    ensure_built()
    inp = wl.make_attention_inputs(
        batch=3, q_len=q_len, num_q_heads=24, num_kv_heads=4, head_dim=256,
        page_size=ps, prefix_lens=[9000, 700, 20000], kv_dtype=kv_dtype,
        seed=71 + q_len + ps, device=DEV)
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"],
                       checked=True)
    ws = sv.alloc_workspace(sv.verify_workspace_size(desc), DEV)
    sv.set_wait_limit(200)  # SM clock cycles: the first waits run out
    try:
        _call(inp, ws)
        torch.cuda.synchronize()
    finally:
        sv.set_wait_limit(0)
    status = sv.verify_status(ws)  # reads and clears the status word
    assert status & _native.SPEC_STATUS_TIMEOUT
    # the device, the stream and the workspace stay usable
    out = _call(inp, ws)
    torch.cuda.synchronize()
    assert sv.verify_status(ws) == 0
    assert_attention_close(rows_of(out), oracle_attention(inp),
                           kv_dtype != "bf16", "after a timed-out call")
