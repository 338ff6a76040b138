"""GPU block KV append (through the C ABI) against the oracle: bit-exact
pools, scales, positions and cache locations; then verify attention over
the appended cache against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import (assert_attention_close, ensure_built,
                         oracle_attention, rows_of)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(kv_dtype, ps, prefixes, q_len=8, hkv=4, seed=0, scale_k=3.0):
    B = len(prefixes)
    inp = wl.make_attention_inputs(batch=B, q_len=q_len, num_q_heads=24,
                                   num_kv_heads=hkv, head_dim=256,
                                   page_size=ps, prefix_lens=prefixes,
                                   kv_dtype=kv_dtype, seed=seed, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(seed + 3)
    k_new = (torch.randn((B, q_len, hkv, 256), generator=g, device=DEV)
             * scale_k).to(torch.bfloat16)
    v_new = torch.randn((B, q_len, hkv, 256), generator=g,
                        device=DEV).to(torch.bfloat16)
    return inp, k_new, v_new


def _both(inp, k_new, v_new):
    ensure_built()
    bits = wl.to_numpy_bits
    fp8 = inp["k_scales"] is not None
    ref = oracle.kv_append(
        bits(k_new), bits(v_new), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None)
    B, q_len = k_new.shape[:2]
    pos = torch.full((B, q_len), -7, dtype=torch.int32, device=DEV)
    loc = torch.full((B, q_len), -7, dtype=torch.int64, device=DEV)
    sv.kv_append(k_new, v_new, inp["k_pages"], inp["v_pages"],
                 inp["page_table"], inp["seq_lens"], k_scales=inp["k_scales"],
                 v_scales=inp["v_scales"], positions=pos, cache_loc=loc)
    torch.cuda.synchronize()
    got = [bits(inp["k_pages"]), bits(inp["v_pages"])]
    if fp8:
        got += [bits(inp["k_scales"]), bits(inp["v_scales"])]
    want = [ref[0], ref[1]] + ([ref[2], ref[3]] if fp8 else [])
    for g_, w_ in zip(got, want):
        assert np.array_equal(g_, w_)      # NaN poison compares as bits
    assert np.array_equal(pos.cpu().numpy(), ref[4])
    assert np.array_equal(loc.cpu().numpy(), ref[5])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("ps", [8, 16, 64])
def test_append_bit_exact(kv_dtype, ps):
    inp, k_new, v_new = _case(kv_dtype, ps, [0, 100, 1000, 63],
                              seed=ps + len(kv_dtype))
    _both(inp, k_new, v_new)


def test_fp8_append_special_values():
    inp, k_new, v_new = _case("fp8_e4m3", 16, [20, 5], seed=3)
    k_new[0, 0, 0] = 0.0                        # amax 0 -> scale 1
    k_new[0, 1, 1, :64] = -0.0                  # signed zeros keep the sign
    k_new[1, 2, 0, 64:128] = 1e4                # large block, scale ~22.3
    k_new[1, 3, 2, 5] = 3.0e-5                  # flushes to a zero code
    v_new[1, 0, 3, :] = 2.0 ** -20              # amax/448 rounds to 0 -> 1
    v_new[1, 1, 3, :64] = 2.0 ** -14            # fp16-subnormal scale
    v_new[1, 1, 3, 64:128] = -(2.0 ** -13)
    _both(inp, k_new, v_new)


def test_append_skips_tokens_without_slots_and_reports_bad_pages():
    inp, k_new, v_new = _case("bf16", 16, [40, 300], seed=8)
    inp["seq_lens"][0] = 5                      # 3 block rows before the cache
    t = int(inp["seq_lens"][1]) - 8
    inp["page_table"][1, t // 16] = 1 << 22     # outside the pool
    _both(inp, k_new, v_new)
    ws = sv.alloc_workspace(1024, DEV)
    sv.kv_append(k_new, v_new, inp["k_pages"], inp["v_pages"],
                 inp["page_table"], inp["seq_lens"], checked=True,
                 workspace=ws)
    assert sv.verify_status(ws) == sv._native.SPEC_STATUS_BAD_PAGE


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_append_then_verify_attention(kv_dtype):
    # the cache holds the prefix; the block's K/V arrive through the append
    inp, k_new, v_new = _case(kv_dtype, 64, [3000, 777, 64], seed=21,
                              scale_k=1.0)
    sv.kv_append(k_new, v_new, inp["k_pages"], inp["v_pages"],
                 inp["page_table"], inp["seq_lens"], k_scales=inp["k_scales"],
                 v_scales=inp["v_scales"])
    out = sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                              inp["page_table"], inp["seq_lens"],
                              scale=inp["scale"], k_scales=inp["k_scales"],
                              v_scales=inp["v_scales"])
    torch.cuda.synchronize()
    ref = oracle_attention(inp)
    assert_attention_close(rows_of(out), ref, kv_dtype != "bf16",
                           f"append then attend ({kv_dtype})")
