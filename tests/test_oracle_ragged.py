"""Pins for the oracle's per-request verify widths, commit lengths and
next-block preparation (no GPU).

Ragged attention is checked against torch float64 scaled-dot-product
attention with masks built here from the block layout; accept against a
numpy brute force; the width policies against traces worked by hand from
their stated rules; and the whole accept -> commit -> prepare loop against
serial greedy decoding of a toy target."""
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_target_gb300 import workloads as wl


def _inputs(B, q_max, q_lens, prefix, hq=6, hkv=2, d=64, ps=4,
            kv_dtype="bf16", seed=5):
    # seq_len = prefix + q_b: the block's own rows sit at the cache's end
    inp = wl.make_attention_inputs(
        batch=B, q_len=q_max, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
        page_size=ps, prefix_lens=[p + q - q_max for p, q in
                                   zip(prefix, q_lens)],
        kv_dtype=kv_dtype, seed=seed)
    inp["q_lens"] = torch.tensor(q_lens, dtype=torch.int32)
    return inp


def _oracle(inp, **kw):
    bits = wl.to_numpy_bits
    fp8 = inp["k_scales"] is not None
    return oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].numpy(), inp["seq_lens"].numpy(),
        num_kv_heads=inp["num_kv_heads"], scale=inp["scale"],
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None,
        q_lens=inp["q_lens"].numpy(), **kw)


def _dense(inp, b, which):
    pages = inp[which + "_pages"]
    ps = pages.shape[2]
    L = int(inp["seq_lens"][b])
    ids = inp["page_table"][b, :math.ceil(L / ps)].long()
    x = pages[ids]
    if inp["k_scales"] is None:
        xf = x.to(torch.float64)
    else:
        sc = inp[which + "_scales"][ids].to(torch.float64)
        xf = x.view(torch.float8_e4m3fn).to(torch.float64) * \
            sc.repeat_interleave(64, dim=-1)
    return xf.permute(1, 0, 2, 3).reshape(x.shape[1], -1, x.shape[3])[:, :L]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_ragged_attention_matches_sdpa_with_per_request_masks(kv_dtype):
    q_max, q_lens, prefix = 8, [8, 3, 1, 0, 5], [20, 33, 7, 12, 2]
    inp = _inputs(5, q_max, q_lens, prefix, kv_dtype=kv_dtype,
                  d=64 if kv_dtype == "bf16" else 128)
    inp["q"][3] = float("nan")          # an idle request's rows are unread
    inp["q"][1, 3:] = float("nan")      # so are rows past q_b
    ours = _oracle(inp).reshape(5, q_max, 6, -1)
    q = inp["q"].to(torch.float64)
    for b, qb in enumerate(q_lens):
        assert np.all(ours[b, qb:] == 0.0)
        if qb == 0:
            continue
        L = int(inp["seq_lens"][b])
        k = _dense(inp, b, "k").repeat_interleave(3, dim=0)
        v = _dense(inp, b, "v").repeat_interleave(3, dim=0)
        # block row i is token L - qb + i and sees keys 0 .. L - qb + i
        mask = torch.arange(L)[None, :] <= (L - qb + torch.arange(qb))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b, :qb].transpose(0, 1), k, v, attn_mask=mask,
            scale=inp["scale"]).transpose(0, 1).numpy()
        np.testing.assert_allclose(ours[b, :qb], ref, rtol=1e-11, atol=1e-12)


def test_ragged_rows_equal_a_uniform_block_of_that_width():
    q_max, q_lens, prefix = 6, [2, 6, 4], [40, 9, 17]
    inp = _inputs(3, q_max, q_lens, prefix, seed=9)
    ours = _oracle(inp).reshape(3, q_max, 6, -1)
    bits = wl.to_numpy_bits
    for b, qb in enumerate(q_lens):
        uni = oracle.verify_attention(
            bits(inp["q"][b:b + 1, :qb]), bits(inp["k_pages"]),
            bits(inp["v_pages"]), inp["page_table"][b:b + 1].numpy(),
            inp["seq_lens"][b:b + 1].numpy(), num_kv_heads=2,
            scale=inp["scale"]).reshape(qb, 6, -1)
        assert np.array_equal(ours[b, :qb], uni)


def test_ragged_append_writes_only_the_request_rows():
    q_max, q_lens, prefix = 5, [5, 2, 0, 1], [6, 9, 4, 0]
    inp = _inputs(4, q_max, q_lens, prefix, hkv=2, d=64, ps=4, seed=2)
    bits = wl.to_numpy_bits
    g = torch.Generator().manual_seed(1)
    kn = torch.randn((4, q_max, 2, 64), generator=g).to(torch.bfloat16)
    vn = torch.randn((4, q_max, 2, 64), generator=g).to(torch.bfloat16)
    kp0, vp0 = bits(inp["k_pages"]), bits(inp["v_pages"])
    kp, vp, _, _, pos, loc = oracle.kv_append(
        bits(kn), bits(vn), kp0, vp0, inp["page_table"].numpy(),
        inp["seq_lens"].numpy(), q_lens=np.array(q_lens, np.int32))
    pt = inp["page_table"].numpy()
    expect_k, expect_v = kp0.copy(), vp0.copy()
    for b, qb in enumerate(q_lens):
        L = int(inp["seq_lens"][b])
        for i in range(q_max):
            if i >= qb:
                assert pos[b, i] == -1 and loc[b, i] == -1
                continue
            t = L - qb + i
            page, slot = pt[b, t // 4], t % 4
            assert pos[b, i] == t and loc[b, i] == page * 4 + slot
            expect_k[page, :, slot] = bits(kn)[b, i]
            expect_v[page, :, slot] = bits(vn)[b, i]
    assert np.array_equal(kp, expect_k) and np.array_equal(vp, expect_v)


def _brute_accept(logits, drafts, q_lens, seq_lens):
    B, q_max = drafts.shape
    am = np.argmax(logits, axis=1).reshape(B, q_max)   # lowest index on ties
    acc, nxt, new = [], [], []
    for b in range(B):
        qb = q_lens[b]
        if qb == 0:
            acc.append(0), nxt.append(-1), new.append(seq_lens[b])
            continue
        a = 0
        for j in range(1, qb):
            if drafts[b, j] != am[b, j - 1]:
                break
            a += 1
        acc.append(a), nxt.append(am[b, a]), new.append(seq_lens[b] - qb + a + 1)
    return np.array(acc), np.array(nxt), np.array(new)


def test_ragged_accept_and_new_seq_lens_match_brute_force():
    rng = np.random.default_rng(4)
    B, q_max, V = 9, 8, 50
    q_lens = np.array([8, 1, 0, 3, 8, 5, 2, 7, 4], np.int32)
    seq_lens = rng.integers(10, 1000, size=B).astype(np.int32)
    logits = rng.normal(size=(B * q_max, V)).astype(np.float32)
    am = np.argmax(logits, axis=1).reshape(B, q_max)
    drafts = rng.integers(0, V, size=(B, q_max)).astype(np.int32)
    for b in range(B):                      # plant runs of matches
        run = rng.integers(0, q_max)
        for j in range(1, run + 1):
            drafts[b, j] = am[b, j - 1]
    drafts[1, 1:] = am[1, :-1]              # matches past q_b do not count
    r = oracle.greedy_accept(logits, drafts, q_lens=q_lens, seq_lens=seq_lens)
    acc, nxt, new = _brute_accept(logits, drafts, q_lens, seq_lens)
    assert np.array_equal(r["accept_len"], acc)
    assert np.array_equal(r["next_token"], nxt)
    assert np.array_equal(r["new_seq_lens"], new)
    assert r["accept_len"][1] == 0 and r["new_seq_lens"][1] == seq_lens[1]
    for b in range(B):
        a = acc[b]
        toks = r["out_tokens"][b]
        if q_lens[b] == 0:
            assert np.all(toks == -1)
        else:
            assert np.array_equal(toks[:a], drafts[b, 1:a + 1])
            assert toks[a] == nxt[b] and np.all(toks[a + 1:] == -1)


def _trace(policy, q_max, q0, state0, accepts, **kw):
    widths, q, st = [], q0, np.array([state0], np.float32)
    pt = np.zeros((1, 64), np.int32)
    for a in accepts:
        assert a <= q - 1
        r = oracle.prepare_next_block(policy, q_max, [q], [a], [7], [100],
                                      st, pt, page_size=16, num_pages=1, **kw)
        st = r["state"]
        q = int(r["next_q_lens"][0])
        widths.append(q)
    return widths


def test_doubling_policy_trace():
    # K starts at 1 (width 2), doubles after a fully accepted block, halves
    # after a rejection, and stays within 1 <= K <= q_max - 1 = 4
    widths = _trace("doubling", 5, 2, 1.0, [1, 2, 4, 1, 0, 0, 1])
    assert widths == [3, 5, 5, 3, 2, 2, 3]


def test_ewma_policy_trace():
    # alpha 1/2, width ceil(e + 1.5) in [2, 8], e starting at 7: fully
    # accepted blocks of 8 stay at 8, rejections walk the width down to the
    # floor of two, acceptance brings it back
    widths = _trace("ewma", 8, 8, 7.0,
                    [7, 7, 0, 0, 3, 3, 4, 0, 0, 0, 0])
    assert widths == [8, 8, 5, 4, 4, 5, 5, 4, 3, 2, 2]


def test_ewma_policy_trace_with_quarter_weight():
    # alpha 1/4 keeps 3/4 of the old value: 7 -> 5.25 -> 3.9375 ->
    # (2.953125 + 1.25) -> 3.15234375, all exact in float32
    widths = _trace("ewma", 8, 8, 7.0, [0, 0, 5, 0], alpha=0.25)
    assert widths == [7, 6, 6, 5]


def test_fixed_policy_and_idle_requests():
    pt = np.arange(8, dtype=np.int32).reshape(2, 4)
    r = oracle.prepare_next_block(
        "fixed", 4, [4, 0], [2, 0], [11, -1], [9, 5],
        np.array([0, 0], np.float32), pt, page_size=4, num_pages=8,
        mask_id=99)
    assert r["next_q_lens"].tolist() == [4, 0]
    assert r["next_seq_lens"].tolist() == [13, 5]
    assert r["block_ids"].tolist() == [[11, 99, 99, 99], [-1] * 4]
    assert r["positions"].tolist() == [[9, 10, 11, 12], [-1] * 4]
    # token 9 -> page_table[0, 2] = 2, slot 1 -> 9; token 12 -> page 3
    assert r["cache_loc"].tolist() == [[9, 10, 11, 12], [-1] * 4]
    assert r["missing"] == 0


def test_unreserved_slots_are_counted_not_invented():
    pt = np.array([[5, 3, -1, 70]], np.int32)       # page 2 unreserved
    r = oracle.prepare_next_block("fixed", 6, [6], [5], [1], [6],
                                  np.zeros(1, np.float32), pt, page_size=4,
                                  num_pages=8)
    # tokens 6,7 -> page 3 (slots 2,3); 8..11 -> page table entry -1
    assert r["cache_loc"].tolist() == [[14, 15, -1, -1, -1, -1]]
    assert r["missing"] == 4


@pytest.mark.parametrize("policy", ["fixed", "ewma", "doubling"])
def test_accept_commit_prepare_loop_equals_serial_greedy(policy):
    """Three requests decode side by side through the whole loop: ragged
    verify blocks, accept with commit lengths, and the next-block layout
    from prepare_next_block.  Each request's committed stream must equal
    serial greedy decoding, and every length, position and cache slot the
    loop produces must agree with where the tokens sit in that stream."""
    V, q_max, ps, n_tok = 16, 8, 4, 160
    rng = np.random.default_rng({"fixed": 1, "ewma": 2, "doubling": 3}[policy])
    table = rng.integers(0, V, size=(V, V))

    def target_next(ctx):
        return int(table[ctx[-2] if len(ctx) > 1 else 0, ctx[-1]])

    B, hit = 3, [0.95, 0.6, 0.1]
    streams = [[3 + b] for b in range(B)]
    # the loop runs until the slowest stream has n_tok tokens; the fastest
    # commits up to q_max per step meanwhile
    cap = q_max * (n_tok + 2)
    serial = []
    for b in range(B):
        s = [3 + b]
        while len(s) < cap:
            s.append(target_next(s))
        serial.append(s)
    max_pages = cap // ps + 1
    pt = np.stack([rng.permutation(B * max_pages)[:max_pages]
                   for _ in range(B)]).astype(np.int32)
    kv_len = np.zeros(B, np.int32)            # the boundary has no KV yet
    state = np.array([q_max - 1.0 if policy == "ewma" else 1.0] * B,
                     np.float32)
    q_lens = np.array([q_max if policy != "doubling" else 2] * B, np.int32)
    widths = [[] for _ in range(B)]
    while min(len(s) for s in streams) < n_tok:
        drafts = rng.integers(0, V, size=(B, q_max)).astype(np.int32)
        logits = rng.normal(size=(B * q_max, V)).astype(np.float32)
        for b in range(B):
            qb = int(q_lens[b])
            drafts[b, 0] = streams[b][-1]
            ctx = list(streams[b])
            for j in range(qb):
                t = target_next(ctx)
                logits[b * q_max + j, t] = 50.0
                if j + 1 < qb:
                    d = t if rng.random() < hit[b] else int(rng.integers(0, V))
                    drafts[b, j + 1] = d
                    ctx.append(d)
        seq_lens = kv_len + q_lens
        r = oracle.greedy_accept(logits, drafts, q_lens=q_lens,
                                 seq_lens=seq_lens)
        for b in range(B):
            a = int(r["accept_len"][b])
            streams[b].extend(r["out_tokens"][b, :a + 1].tolist())
            widths[b].append(int(q_lens[b]))
            # the cache now holds every committed token but the bonus
            assert r["new_seq_lens"][b] == len(streams[b]) - 1
        p = oracle.prepare_next_block(
            policy, q_max, q_lens, r["accept_len"], r["next_token"],
            r["new_seq_lens"], state, pt, page_size=ps,
            num_pages=B * max_pages, mask_id=V)
        for b in range(B):
            w = int(p["next_q_lens"][b])
            pos0 = len(streams[b]) - 1          # the bonus token's index
            assert 1 <= w <= q_max
            assert p["next_seq_lens"][b] == pos0 + w
            assert p["block_ids"][b, 0] == streams[b][-1]
            assert np.all(p["block_ids"][b, 1:w] == V)
            assert np.all(p["block_ids"][b, w:] == -1)
            for i in range(w):
                t = pos0 + i
                assert p["positions"][b, i] == t
                assert p["cache_loc"][b, i] == pt[b, t // ps] * ps + t % ps
        assert p["missing"] == 0
        state, q_lens, kv_len = p["state"], p["next_q_lens"], \
            r["new_seq_lens"]
    for b in range(B):
        assert streams[b] == serial[b][:len(streams[b])]
    if policy == "fixed":
        assert all(w == q_max for ws in widths for w in ws)
    else:   # an accurate drafter verifies wider blocks than a poor one
        assert np.mean(widths[0]) > np.mean(widths[2]) + 2
