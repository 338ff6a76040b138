"""FP8 verify attention with K and V^T as tensor-memory operands (blocks of at
most 64 rows per KV head) against the CPU float64 oracle.

The transposed kernel keeps one running maximum per query row shared by 128
token threads, masks per (token lane, row column), and comes in four
instances (N = 16, 32, 48, 64 rows); each case below reaches one of those
paths.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import (assert_attention_close, ensure_built, gpu_attention,
                         oracle_attention, rows_of)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(prefixes, q_len, ps, hq=24, hkv=4, seed=0):
    return wl.make_attention_inputs(
        batch=len(prefixes), q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
        head_dim=256, page_size=ps, prefix_lens=prefixes, kv_dtype="fp8_e4m3",
        seed=seed, device=DEV)


@pytest.mark.parametrize("hq,hkv,q_len,ps", [
    (24, 4, 1, 64),    # 6 rows: N = 16
    (24, 4, 4, 16),    # 24 rows: N = 32
    (24, 4, 5, 128),   # 30 rows: N = 32
    (24, 4, 8, 32),    # 48 rows: N = 48
    (24, 4, 10, 64),   # 60 rows: N = 64
    (32, 4, 8, 8),     # 64 rows, 8-token pages: 16 boxes per tile
    (8, 4, 8, 16),     # 16 rows: N = 16
])
def test_fp8_row_counts_and_page_sizes(hq, hkv, q_len, ps):
    # prefixes with whole, partial and single-unit tiles, one empty prefix
    inp = _case([0, 130, 1000, 257, 4099], q_len, ps, hq=hq, hkv=hkv,
                seed=hq * 100 + q_len * 10 + ps)
    out = gpu_attention(inp)
    assert_attention_close(rows_of(out), oracle_attention(inp), True,
                           f"Hq={hq} Hkv={hkv} q_len={q_len} ps={ps}")


def test_fp8_running_max_jumps_mid_sequence():
    # the second half of every sequence has 8x larger keys, so the row
    # maxima jump by far more than 2^8 partway through a piece: O^T and the
    # partial row sums are rescaled while later tiles are in flight
    inp = _case([3000, 700, 129, 6000], 8, 64, seed=77)
    ks = inp["k_scales"]
    pt = inp["page_table"].cpu()
    lens = inp["seq_lens"].cpu().tolist()
    for b, n in enumerate(lens):
        npg = (n + 63) // 64
        for pi in range(npg // 2, npg):
            ks[int(pt[b, pi])] *= 8
    out = gpu_attention(inp)
    assert_attention_close(rows_of(out), oracle_attention(inp), True,
                           "fp8 running max jump")


@pytest.mark.parametrize("lane,mult", [(40, 256.0), (127, 256.0), (5, 4.0)])
def test_fp8_single_token_spike(lane, mult):
    # One cached token, lane `lane` of a tile in the middle of each request's
    # prefix, gets keys `mult` times larger, so only the warp holding that
    # lane sees its scores pass the running maxima.  The four softmax warps
    # must agree to raise them for that tile.  At 256x the scores pass the
    # maxima by far more than fp16 and fp32 exp2 can hold, so the first P^T
    # written for the tile overflows and must be replaced before PV reads
    # it.  At 4x the jump lands near the rescale threshold: past it for some
    # rows, short of it for others.
    inp = _case([3000, 6000, 1500], 8, 64, seed=91 + lane)
    ks = inp["k_scales"]
    pt = inp["page_table"].cpu()
    for b, n in enumerate(inp["seq_lens"].cpu().tolist()):
        t = (n // 2) // 128 * 128 + lane
        ks[int(pt[b, t // 64]), :, t % 64, :] *= mult
    out = gpu_attention(inp)
    assert torch.isfinite(out.float()).all()
    assert_attention_close(rows_of(out), oracle_attention(inp), True,
                           f"fp8 spike lane {lane} x{mult}")


def test_fp8_ragged_widths():
    inp = _case([700, 70, 1500, 5, 333], 8, 64, seed=48)
    ql = torch.tensor([8, 5, 1, 0, 3], dtype=torch.int32, device=DEV)
    ensure_built()
    out = sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                              inp["page_table"], inp["seq_lens"],
                              scale=inp["scale"], k_scales=inp["k_scales"],
                              v_scales=inp["v_scales"], q_lens=ql)
    torch.cuda.synchronize()
    bits = wl.to_numpy_bits
    ref = oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        num_kv_heads=4, scale=inp["scale"], k_scales=bits(inp["k_scales"]),
        v_scales=bits(inp["v_scales"]), q_lens=ql.cpu().numpy())
    assert_attention_close(rows_of(out), ref, True, "fp8 ragged widths")
    o = out.float().view(5, 8, 24, 256)
    assert torch.all(o[3] == 0)          # q_b = 0: every row zero
    assert torch.all(o[1, 5:] == 0) and torch.all(o[4, 3:] == 0)


def test_fp8_error_well_inside_the_bound():
    # fp16 dequantised operands and fp16 P: the error is a few 1e-3, far
    # from the 5e-2 bound, on a long single request split over many CTAs
    inp = _case([20000], 8, 64, seed=5)
    out = gpu_attention(inp)
    err = np.abs(rows_of(out).astype(np.float64) - oracle_attention(inp))
    assert err.max() < 1e-2, err.max()


def test_fp8_bad_page_id_sets_status_without_fault():
    inp = _case([500], 8, 16, seed=4)
    inp["page_table"][0, 3] = 1 << 20      # outside the pool
    ensure_built()
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"],
                       checked=True)
    ws = sv.alloc_workspace(sv.verify_workspace_size(desc), DEV)
    kw = dict(scale=inp["scale"], k_scales=inp["k_scales"],
              v_scales=inp["v_scales"], checked=True, workspace=ws)
    sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                        inp["page_table"], inp["seq_lens"], **kw)
    assert sv.verify_status(ws) == sv._native.SPEC_STATUS_BAD_PAGE
    inp["page_table"][0, 3] = 0
    sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                        inp["page_table"], inp["seq_lens"], **kw)
    assert sv.verify_status(ws) == 0


def test_fp8_repeatable_and_independent_of_workspace():
    inp = _case([5000, 17], 8, 64, seed=9)
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"])
    ws = torch.full((sv.verify_workspace_size(desc),), 0xFF,
                    dtype=torch.uint8, device=DEV)
    a = gpu_attention(inp, workspace=ws)
    b = gpu_attention(inp, workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_attention_close(rows_of(a), oracle_attention(inp), True,
                           "fp8 garbage workspace")



def test_fp8_two_slot_instance_under_many_short_pieces():
    # N = 64 keeps two V^T slots, so the two dequant warp sets, which take
    # alternate tiles, write each slot in turn; many short pieces (short
    # mixed-length requests over every SM) make one set run far ahead of
    # the other's PV.  Each set waits on its own slot barriers, so no wait
    # can be taken for a phase two ahead of the barrier.
    g = torch.Generator().manual_seed(64)
    prefixes = torch.randint(60, 900, (24,), generator=g).tolist()
    for hq, q_len, ps in ((32, 8, 16), (24, 10, 64)):
        inp = _case(prefixes, q_len, ps, hq=hq, seed=hq + q_len + ps)
        out = gpu_attention(inp)
        assert_attention_close(rows_of(out), oracle_attention(inp), True,
                               f"two-slot instance Hq={hq} q_len={q_len}")
