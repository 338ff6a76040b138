"""GPU verify attention (through the C ABI) against the CPU float64 oracle."""
import pytest
import torch

from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import (assert_attention_close, gpu_attention,
                         oracle_attention, rows_of)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, q_len, prefix, ps, kv_dtype="bf16", hq=24, hkv=4, seed=0,
          **kw):
    prefixes = [prefix, prefix // 2 + 3, prefix + 5][:B] if B <= 3 else \
        list(prefix)
    return wl.make_attention_inputs(
        batch=B, q_len=q_len, num_q_heads=hq, num_kv_heads=hkv, head_dim=256,
        page_size=ps, prefix_lens=prefixes, kv_dtype=kv_dtype, seed=seed,
        device=DEV, **kw)


def _check_all(inp, what):
    out = gpu_attention(inp)
    ref = oracle_attention(inp)
    assert_attention_close(rows_of(out), ref, inp["k_scales"] is not None,
                           what)
    return out


PREFIXES = [0, 1, 15, 16, 17, 63, 64, 65, 321, 4096]


@pytest.mark.parametrize("q_len", [1, 8, 16])
@pytest.mark.parametrize("pi", range(len(PREFIXES)))
def test_grid_bf16(q_len, pi):
    prefix = PREFIXES[pi]
    ps = 16 if pi % 2 == 0 else 64
    B = 1 if pi % 3 == 0 else 3
    inp = _case(B, q_len, prefix, ps, seed=100 * q_len + pi)
    _check_all(inp, f"q_len={q_len} prefix={prefix} ps={ps} B={B}")


FP8_PREFIXES = [0, 17, 65, 321, 4096]


@pytest.mark.parametrize("q_len", [1, 8, 16])
@pytest.mark.parametrize("pi", range(len(FP8_PREFIXES)))
def test_grid_fp8(q_len, pi):
    prefix = FP8_PREFIXES[pi]
    ps = 16 if pi % 2 == 0 else 64
    B = 1 if pi % 3 == 0 else 3
    inp = _case(B, q_len, prefix, ps, kv_dtype="fp8_e4m3",
                seed=500 + 10 * q_len + pi)
    _check_all(inp, f"fp8 q_len={q_len} prefix={prefix} ps={ps} B={B}")


@pytest.mark.parametrize("ps", [8, 32, 128])
def test_fp8_page_sizes_and_ragged(ps):
    g = torch.Generator().manual_seed(ps)
    prefixes = torch.randint(0, 2500, (9,), generator=g).tolist()
    inp = _case(9, 8, prefixes, ps, kv_dtype="fp8_e4m3", seed=ps + 7)
    _check_all(inp, f"fp8 page_size={ps} ragged")


def test_fp8_rejects_small_pages():
    import speculative_decoding_target_gb300 as sv
    inp = _case(1, 8, 40, 4, kv_dtype="fp8_e4m3", seed=1)
    with pytest.raises(sv.SpecError) as e:     # refused on the host
        gpu_attention(inp)
    assert "page_size" in str(e.value)


@pytest.mark.parametrize("hq,hkv,q_len", [(8, 8, 8), (32, 4, 16), (4, 1, 16),
                                          (24, 4, 3), (12, 2, 5)])
def test_gqa_shapes(hq, hkv, q_len):
    inp = _case(2, q_len, 200, 16, hq=hq, hkv=hkv, seed=hq + q_len)
    _check_all(inp, f"Hq={hq} Hkv={hkv} q_len={q_len}")


@pytest.mark.parametrize("ps", [1, 4, 128, 256])
def test_page_sizes(ps):
    inp = _case(2, 8, 300, ps, seed=ps)
    _check_all(inp, f"page_size={ps}")


@pytest.mark.parametrize("B,hq,hkv", [(1, 4, 1), (2, 24, 4), (4, 24, 4)])
def test_merge_batches_with_a_late_dominant_key(B, hq, hkv):
    # Few (request, KV head) segments over the whole grid: one segment split
    # ~100 ways (the merge's 20-split batches, several rounds per warp), 8
    # segments ~19 ways (12-split batches) and 16 segments (8-split
    # batches).  One key near the end of every sequence is scaled up, so the
    # largest log-sum-exp sits in a late split and each warp's running
    # maximum has to grow after it has summed earlier splits.
    prefix = 20000 if B <= 3 else [20000, 12003, 20005, 7000][:B]
    inp = _case(B, 16, prefix, 64, hq=hq, hkv=hkv, seed=300 + B)
    pt = inp["page_table"].cpu()
    for b, n in enumerate(inp["seq_lens"].cpu().tolist()):
        t = n - 40
        inp["k_pages"][int(pt[b, t // 64]), :, t % 64, :] *= 8
    _check_all(inp, f"merge batches B={B} Hkv={hkv}")


def test_many_ragged_requests_exercise_the_plan():
    g = torch.Generator().manual_seed(5)
    prefixes = torch.randint(0, 3000, (40,), generator=g).tolist()
    prefixes[3] = 0
    prefixes[7] = 64 * 20 - 8
    inp = _case(40, 8, prefixes, 64, seed=77)
    _check_all(inp, "40 ragged requests")


def test_short_and_empty_windows_give_zero_rows():
    # seq_len < q_len: rows whose causal window is empty output zeros;
    # seq_len = 0: every row of that request is zero.
    inp = _case(3, 8, 10, 16, seed=3)
    inp["seq_lens"] = torch.tensor([5, 0, 8], dtype=torch.int32, device=DEV)
    out = _check_all(inp, "short windows")
    o = out.float().view(3, 8, 24, 256)
    assert torch.all(o[0, :3] == 0) and torch.any(o[0, 3:] != 0)
    assert torch.all(o[1] == 0)


def test_result_independent_of_workspace_contents_and_repeatable():
    inp = _case(2, 16, 5000, 64, seed=9)
    import speculative_decoding_target_gb300 as sv
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"])
    ws = torch.full((sv.verify_workspace_size(desc),), 0xFF,
                    dtype=torch.uint8, device=DEV)   # NaN-patterned garbage
    a = gpu_attention(inp, workspace=ws)
    b = gpu_attention(inp, workspace=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = oracle_attention(inp)
    assert_attention_close(rows_of(a), ref, False, "garbage workspace")


def test_bad_page_id_sets_status_without_fault():
    import speculative_decoding_target_gb300 as sv
    inp = _case(1, 8, 500, 16, seed=4)
    inp["page_table"][0, 3] = 1 << 20      # outside the pool
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"],
                       checked=True)
    ws = sv.alloc_workspace(sv.verify_workspace_size(desc), DEV)
    sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                        inp["page_table"], inp["seq_lens"],
                        scale=inp["scale"], checked=True, workspace=ws)
    assert sv.verify_status(ws) == sv._native.SPEC_STATUS_BAD_PAGE
    # a clean call afterwards reports nothing
    inp["page_table"][0, 3] = 0
    sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                        inp["page_table"], inp["seq_lens"],
                        scale=inp["scale"], checked=True, workspace=ws)
    assert sv.verify_status(ws) == 0


@pytest.mark.parametrize("name", wl.WORKLOAD_ORDER)
def test_full_size_workloads_every_row(name):
    """Every attention row of each full-size workload, in the launch
    configuration the benchmark times (the whole batch in one call, the
    device-side split plan over every SM), element by element against the
    oracle."""
    w = wl.WORKLOADS[name]
    fp8 = w.kv_dtype != "bf16"
    inp = wl.workload_inputs(w, device=DEV, with_accept=False)
    out = gpu_attention(inp)
    torch.cuda.synchronize()
    # property at any size: every output is a convex combination of V rows
    if fp8:
        v = inp["v_pages"].view(torch.float8_e4m3fn).float() * \
            inp["v_scales"].float().repeat_interleave(64, dim=-1)
    else:
        v = inp["v_pages"].float()
    vmax = v.nan_to_num(0.0).abs().max().item()
    del v
    o = out.float()
    assert torch.isfinite(o).all()
    assert o.abs().max().item() <= vmax * (1 + 2 ** -7) + (0.05 if fp8 else 0)
    n_rows = w.batch * w.q_len * w.num_q_heads
    ref = oracle_attention(inp)
    assert ref.shape == (n_rows, w.head_dim)
    assert_attention_close(rows_of(out), ref, fp8,
                           f"{name}: all {n_rows} rows")


def test_hundreds_of_tiny_requests():
    # many segments: the plan's prefix over the batch, phantom-only CTAs,
    # split slots across hundreds of (request, head) segments
    g = torch.Generator().manual_seed(17)
    prefixes = torch.randint(0, 90, (600,), generator=g).tolist()
    prefixes[0] = 0
    inp = _case(600, 8, prefixes, 16, seed=600)
    _check_all(inp, "600 tiny requests")


def test_every_sequence_empty_gives_zero_output():
    inp = _case(5, 8, [40, 0, 7, 100, 3], 16, seed=8)
    inp["seq_lens"] = torch.zeros(5, dtype=torch.int32, device=DEV)
    out = gpu_attention(inp)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0)


def test_fp8_widest_tile_with_ragged_widths():
    # q_len 16 x group 8 = 128 rows, every TMEM lane in use
    inp = _case(4, 16, [700, 70, 1500, 5], 64, kv_dtype="fp8_e4m3", hq=32,
                hkv=4, seed=128)
    import speculative_decoding_target_gb300 as sv
    ql = torch.tensor([16, 9, 1, 0], dtype=torch.int32, device=DEV)
    out = sv.verify_attention(inp["q"], inp["k_pages"], inp["v_pages"],
                              inp["page_table"], inp["seq_lens"],
                              scale=inp["scale"], k_scales=inp["k_scales"],
                              v_scales=inp["v_scales"], q_lens=ql)
    torch.cuda.synchronize()
    bits = wl.to_numpy_bits
    import oracle
    ref = oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        num_kv_heads=4, scale=inp["scale"], k_scales=bits(inp["k_scales"]),
        v_scales=bits(inp["v_scales"]), q_lens=ql.cpu().numpy())
    assert_attention_close(rows_of(out), ref, True, "fp8 128-row tile")
