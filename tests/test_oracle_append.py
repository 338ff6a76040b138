"""Pins for the oracle's encoders and its block KV append (no GPU).

The encoders are checked against library conversions (torch float8_e4m3fn,
numpy float16) and by round trips over every code; the append is checked
against closed forms (positions, cache locations, copies) and, for FP8,
against the stated scale rule evaluated with numpy's float32 division and
float16 cast plus torch's E4M3 conversion."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_target_gb300 import workloads as wl


def _torch_e4m3(x):
    t = torch.from_numpy(np.asarray(x, np.float32)).clamp(-448, 448)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_matches_torch_and_round_trips():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.normal(size=20000) * 50, rng.normal(size=5000) * 2.0 ** -7,
        rng.uniform(-600, 600, 5000),
        oracle.decode_e4m3(np.arange(256)).astype(np.float32)]).astype(np.float32)
    x = x[np.isfinite(x)]
    # midpoints between neighbouring codes: ties go to the even code
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    v = oracle.decode_e4m3(codes)
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    assert np.array_equal(oracle.encode_e4m3(x), _torch_e4m3(x))
    finite = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], np.uint8)
    back = oracle.encode_e4m3(oracle.decode_e4m3(finite).astype(np.float32))
    assert np.array_equal(back, finite)
    assert oracle.encode_e4m3(np.array([1e9, -1e9, np.inf], np.float32)).tolist() \
        == [0x7E, 0xFE, 0x7E]


def test_fp16_encoder_matches_numpy():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(size=50000) * 1e3, rng.normal(size=20000) * 1e-5,
                        rng.uniform(-7e4, 7e4, 5000),
                        np.array([0.0, -0.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                                  65504, 65519.99, 65520, 1e30])]).astype(np.float32)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.encode_fp16(x), ref)


def _append_case(kv_dtype, ps, B=3, q_len=5, hkv=2, d=128, seed=0):
    prefixes = [0, 13, 40][:B]
    inp = wl.make_attention_inputs(batch=B, q_len=q_len, num_q_heads=hkv,
                                   num_kv_heads=hkv, head_dim=d, page_size=ps,
                                   prefix_lens=prefixes, kv_dtype=kv_dtype,
                                   seed=seed)
    g = torch.Generator().manual_seed(seed + 9)
    k_new = (torch.randn((B, q_len, hkv, d), generator=g) * 3).to(torch.bfloat16)
    v_new = (torch.randn((B, q_len, hkv, d), generator=g)).to(torch.bfloat16)
    return inp, k_new, v_new


def _run(inp, k_new, v_new):
    bits = wl.to_numpy_bits
    fp8 = inp["k_scales"] is not None
    return oracle.kv_append(
        bits(k_new), bits(v_new), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].numpy(), inp["seq_lens"].numpy(),
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None)


@pytest.mark.parametrize("ps", [1, 4, 16])
def test_bf16_append_copies_rows_and_reports_positions(ps):
    inp, k_new, v_new = _append_case("bf16", ps)
    kp, vp, _, _, pos, loc = _run(inp, k_new, v_new)
    kp0 = wl.to_numpy_bits(inp["k_pages"])
    sl = inp["seq_lens"].numpy()
    pt = inp["page_table"].numpy()
    touched = np.zeros(kp0.shape[:3], bool)
    for b in range(3):
        for i in range(5):
            t = sl[b] - 5 + i
            assert pos[b, i] == t
            page, slot = pt[b, t // ps], t % ps
            assert loc[b, i] == page * ps + slot
            for g in range(2):
                assert np.array_equal(kp[page, g, slot],
                                      wl.to_numpy_bits(k_new[b, i, g]))
                assert np.array_equal(vp[page, g, slot],
                                      wl.to_numpy_bits(v_new[b, i, g]))
                touched[page, g, slot] = True
    assert np.array_equal(kp[~touched], kp0[~touched])   # nothing else moved


def test_fp8_append_follows_the_scale_rule():
    inp, k_new, v_new = _append_case("fp8_e4m3", 16, d=256)
    kp, vp, ks, vs, pos, loc = _run(inp, k_new, v_new)
    ps = 16
    for b in range(3):
        for i in range(5):
            page, slot = divmod(int(loc[b, i]), ps)
            for g in range(2):
                for new, pool, sc in ((k_new, kp, ks), (v_new, vp, vs)):
                    x = new[b, i, g].float().numpy().reshape(4, 64)
                    amax = np.abs(x).max(axis=1).astype(np.float32)
                    s = (amax / np.float32(448)).astype(np.float16)
                    s[s == 0] = np.float16(1)
                    assert np.array_equal(sc[page, g, slot], s.view(np.uint16))
                    y = x / s.astype(np.float32)[:, None]
                    assert np.array_equal(pool[page, g, slot],
                                          _torch_e4m3(y.astype(np.float32)).ravel())
                    # decoding the stored block gives x back to within half
                    # an E4M3 step of the scaled value
                    dq = oracle.decode_e4m3(pool[page, g, slot]).reshape(4, 64) \
                        * s.astype(np.float64)[:, None]
                    bound = np.abs(x) * 2.0 ** -4 + s.astype(np.float64)[:, None] * 2.0 ** -10
                    assert np.all(np.abs(dq - x) <= bound + 1e-12)


def test_append_then_attention_equals_a_prefilled_pool():
    # appending the block to a pool equals generating the pool with it
    inp, k_new, v_new = _append_case("bf16", 4, hkv=2, d=64)
    kp, vp, _, _, _, _ = _run(inp, k_new, v_new)
    q = (torch.randn((3, 5, 4, 64), generator=torch.Generator().manual_seed(5))
         ).to(torch.bfloat16)
    bits = wl.to_numpy_bits
    a = oracle.verify_attention(bits(q), kp, vp, inp["page_table"].numpy(),
                                inp["seq_lens"].numpy(), num_kv_heads=2,
                                scale=0.125)
    # the block's rows written straight into the pool tensors
    k2, v2 = inp["k_pages"].clone(), inp["v_pages"].clone()
    sl, pt = inp["seq_lens"], inp["page_table"]
    for b in range(3):
        for i in range(5):
            t = int(sl[b]) - 5 + i
            k2[int(pt[b, t // 4]), :, t % 4] = k_new[b, i]
            v2[int(pt[b, t // 4]), :, t % 4] = v_new[b, i]
    r = oracle.verify_attention(bits(q), bits(k2), bits(v2), pt.numpy(),
                                sl.numpy(), num_kv_heads=2, scale=0.125)
    assert np.array_equal(a, r)


def test_tokens_without_a_slot_are_skipped():
    inp, k_new, v_new = _append_case("bf16", 4)
    inp["seq_lens"][0] = 3          # rows 0, 1 would sit before the cache
    inp["page_table"][2, 10] = 99999   # a bad page id for request 2
    kp, vp, _, _, pos, loc = _run(inp, k_new, v_new)
    assert pos[0].tolist() == [-1, -1, 0, 1, 2]
    assert loc[0, 0] == -1 and loc[0, 1] == -1 and loc[0, 2] >= 0
    t_bad = [int(inp["seq_lens"][2]) - 5 + i for i in range(5)]
    for i, t in enumerate(t_bad):
        if t // 4 == 10:
            assert loc[2, i] == -1
