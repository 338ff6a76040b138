"""GPU per-request verify widths (through the C ABI) against the oracle:
ragged verify attention within the stated tolerance; ragged KV append,
accept with commit lengths and next-block preparation bit for bit; and a
multi-step accept -> prepare loop kept on the device."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import assert_attention_close, ensure_built, rows_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(q_lens, prefix, q_max=8, ps=16, kv_dtype="bf16", hq=24, hkv=4,
            seed=0):
    inp = wl.make_attention_inputs(
        batch=len(q_lens), q_len=q_max, num_q_heads=hq, num_kv_heads=hkv,
        head_dim=256, page_size=ps, prefix_lens=prefix, kv_dtype=kv_dtype,
        seed=seed, device=DEV)
    inp["q_lens"] = torch.tensor(q_lens, dtype=torch.int32, device=DEV)
    # rows past each block hold NaN: they must never reach an output
    for b, qb in enumerate(q_lens):
        inp["q"][b, qb:] = float("nan")
    return inp


def _oracle_attention(inp, rows=None):
    bits = wl.to_numpy_bits
    fp8 = inp["k_scales"] is not None
    return oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        num_kv_heads=inp["num_kv_heads"], scale=inp["scale"],
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None,
        q_lens=inp["q_lens"].cpu().numpy(), rows=rows)


def _gpu_attention(inp, noalloc=False):
    ensure_built()
    fn = sv._native.verify_attention_noalloc if noalloc else sv.verify_attention
    return fn(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"],
              inp["seq_lens"], scale=inp["scale"], k_scales=inp["k_scales"],
              v_scales=inp["v_scales"], q_lens=inp["q_lens"])


CASES = [  # (q_lens, prefix, q_max, page size, kv dtype)
    ([8, 3, 1, 0, 5, 2], [300, 77, 1000, 40, 5, 0], 8, 16, "bf16"),
    ([16, 9, 2], [4100, 63, 129], 16, 64, "bf16"),
    ([4, 1, 8, 0], [250, 3000, 17, 64], 8, 64, "fp8_e4m3"),
    ([1, 8, 6], [90, 33, 2], 8, 4, "bf16"),        # mma.sync kernel
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_ragged_attention(case):
    q_lens, prefix, q_max, ps, kv = CASES[case]
    inp = _inputs(q_lens, prefix, q_max=q_max, ps=ps, kv_dtype=kv,
                  seed=40 + case)
    out = _gpu_attention(inp)
    torch.cuda.synchronize()
    o = out.float().view(len(q_lens), q_max, -1)
    for b, qb in enumerate(q_lens):
        assert torch.all(o[b, qb:] == 0)
    assert_attention_close(rows_of(out), _oracle_attention(inp), kv != "bf16",
                           f"ragged case {case}")


def test_ragged_attention_without_workspace():
    inp = _inputs([2, 8, 5], [700, 12, 64], seed=3)
    out = _gpu_attention(inp, noalloc=True)
    torch.cuda.synchronize()
    assert_attention_close(rows_of(out), _oracle_attention(inp), False,
                           "ragged, no workspace")


def test_ragged_full_size_sampled_rows():
    w = wl.WORKLOADS["b8_q8_p32k"]
    inp = wl.workload_inputs(w, device=DEV, with_accept=False)
    g = torch.Generator().manual_seed(8)
    ql = torch.randint(0, w.q_len + 1, (w.batch,), generator=g)
    ql[0], ql[1] = w.q_len, 1
    inp["q_lens"] = ql.to(torch.int32).to(DEV)
    out = _gpu_attention(inp)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    total = w.batch * w.q_len * w.num_q_heads
    rows = np.sort(rng.choice(total, 48, replace=False)).astype(np.int64)
    assert_attention_close(rows_of(out, rows),
                           _oracle_attention(inp, rows=rows), False,
                           "b8_q8_p32k ragged")
    o = out.float().view(w.batch, w.q_len, -1)
    for b in range(w.batch):
        assert torch.all(o[b, int(ql[b]):] == 0)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_ragged_append_bit_exact(kv):
    ensure_built()
    q_lens, prefix = [8, 3, 0, 1, 6], [100, 20, 50, 0, 333]
    inp = _inputs(q_lens, prefix, kv_dtype=kv, seed=7)
    B, q_max = len(q_lens), 8
    g = torch.Generator(device=DEV).manual_seed(2)
    kn = torch.randn((B, q_max, 4, 256), generator=g, device=DEV).to(
        torch.bfloat16)
    vn = torch.randn((B, q_max, 4, 256), generator=g, device=DEV).to(
        torch.bfloat16)
    bits = wl.to_numpy_bits
    fp8 = kv != "bf16"
    ref = oracle.kv_append(
        bits(kn), bits(vn), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None, q_lens=q_lens)
    pos = torch.full((B, q_max), -7, dtype=torch.int32, device=DEV)
    loc = torch.full((B, q_max), -7, dtype=torch.int64, device=DEV)
    sv.kv_append(kn, vn, inp["k_pages"], inp["v_pages"], inp["page_table"],
                 inp["seq_lens"], k_scales=inp["k_scales"],
                 v_scales=inp["v_scales"], positions=pos, cache_loc=loc,
                 q_lens=inp["q_lens"])
    torch.cuda.synchronize()
    assert np.array_equal(bits(inp["k_pages"]), ref[0])
    assert np.array_equal(bits(inp["v_pages"]), ref[1])
    if fp8:
        assert np.array_equal(bits(inp["k_scales"]), ref[2])
        assert np.array_equal(bits(inp["v_scales"]), ref[3])
    assert np.array_equal(pos.cpu().numpy(), ref[4])
    assert np.array_equal(loc.cpu().numpy(), ref[5])


def _accept_case(B, q_max, V, seed):
    inp = wl.make_accept_inputs(batch=B, q_len=q_max, vocab=V, accept_p=0.7,
                                seed=seed, device=DEV)
    g = torch.Generator().manual_seed(seed)
    ql = torch.randint(0, q_max + 1, (B,), generator=g).to(torch.int32)
    ql[0] = q_max
    sl = torch.randint(q_max, 100000, (B,), generator=g).to(torch.int32)
    logits = inp["logits"].view(B, q_max, V)
    for b in range(B):           # rows past the block are not read
        logits[b, int(ql[b]):] = float("nan")
    return inp["logits"], inp["draft_ids"], ql.to(DEV), sl.to(DEV)


@pytest.mark.parametrize("B,q_max,V", [(7, 8, 248320), (33, 16, 5000),
                                       (3, 1, 100), (40, 8, 2052),
                                       (1024, 16, 36), (1025, 4, 36)])
def test_accept_commit_bit_exact(B, q_max, V):
    ensure_built()
    logits, drafts, ql, sl = _accept_case(B, q_max, V, seed=B + q_max)
    acc, nxt, toks, new = sv.greedy_accept_commit(logits, drafts, ql, sl)
    torch.cuda.synchronize()
    ref = oracle.greedy_accept(logits.cpu().numpy(), drafts.cpu().numpy(),
                               q_lens=ql.cpu().numpy(),
                               seq_lens=sl.cpu().numpy())
    assert np.array_equal(acc.cpu().numpy(), ref["accept_len"])
    assert np.array_equal(nxt.cpu().numpy(), ref["next_token"])
    assert np.array_equal(toks.cpu().numpy(), ref["out_tokens"])
    assert np.array_equal(new.cpu().numpy(), ref["new_seq_lens"])


@pytest.mark.parametrize("policy", ["fixed", "ewma", "doubling"])
def test_prepare_next_block_bit_exact(policy):
    ensure_built()
    rng = np.random.default_rng(len(policy))
    B, q_max, ps, max_pages, num_pages = 300, 16, 16, 40, 5000
    ql = rng.integers(0, q_max + 1, B).astype(np.int32)
    acc = np.array([rng.integers(0, max(q, 1)) for q in ql], np.int32)
    acc[:40] = np.maximum(ql[:40] - 1, 0)          # fully accepted blocks
    nxt = rng.integers(0, 248320, B).astype(np.int32)
    new = rng.integers(1, 600, B).astype(np.int32)
    if policy == "ewma":    # arbitrary floats exercise the float32 rounding
        state = rng.uniform(0, q_max, B).astype(np.float32)
        kw = dict(alpha=float(np.float32(0.3)), offset=1.5, min_width=2)
    else:
        state = rng.integers(1, q_max, B).astype(np.float32)
        kw = {}
    pt = rng.integers(0, num_pages, (B, max_pages)).astype(np.int32)
    pt[5, 600 // ps:] = -1                          # unreserved tail
    pt[9, 2] = num_pages + 3                        # outside the pool
    ql[5] = ql[9] = 8
    new[5], new[9] = 595, 30                        # both reach those pages
    ref = oracle.prepare_next_block(
        policy, q_max, ql, acc, nxt, new, state, pt, page_size=ps,
        num_pages=num_pages, mask_id=248319, **kw)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    st = t(state)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pol = sv.width_policy(policy, q_max, mask_id=248319, **kw)
    out = sv.prepare_next_block(pol, t(ql), t(acc), t(nxt), t(new), st,
                                t(pt), page_size=ps, num_pages=num_pages,
                                status=status)
    torch.cuda.synchronize()
    for k in ("next_q_lens", "next_seq_lens", "block_ids", "positions",
              "cache_loc"):
        assert np.array_equal(out[k].cpu().numpy(), ref[k]), k
    assert np.array_equal(st.cpu().numpy().view(np.uint32),
                          ref["state"].view(np.uint32))
    assert ref["missing"] > 0
    assert int(status.item()) == sv._native.SPEC_STATUS_NO_SLOT


@pytest.mark.parametrize("policy", ["ewma", "doubling"])
def test_device_loop_matches_oracle_loop(policy):
    """Ten verify steps whose widths, lengths and blocks stay on the device:
    accept-commit then prepare, each step's logits planted so that the
    drafts' fate varies; every device state equals the oracle's."""
    ensure_built()
    B, q_max, V, ps, max_pages = 16, 8, 3000, 16, 64
    rng = np.random.default_rng(5)
    pt = rng.permutation(B * max_pages).reshape(B, max_pages).astype(np.int32)
    pol_kw = dict(alpha=0.5, offset=1.5, min_width=2, mask_id=V)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    state_h = np.full(B, q_max - 1.0 if policy == "ewma" else 1.0, np.float32)
    ql_h = np.full(B, q_max if policy == "ewma" else 2, np.int32)
    kv_h = rng.integers(10, 200, B).astype(np.int32)
    state_d, ql_d, kv_d, pt_d = d(state_h), d(ql_h), d(kv_h), d(pt)
    pol = sv.width_policy(policy, q_max, **pol_kw)
    for step in range(10):
        logits = rng.normal(size=(B * q_max, V)).astype(np.float32)
        am = np.argmax(logits, 1).reshape(B, q_max)
        drafts = rng.integers(0, V, (B, q_max)).astype(np.int32)
        hit = rng.random((B, q_max)) < np.linspace(0.95, 0.2, B)[:, None]
        for b in range(B):
            for j in range(1, q_max):
                if hit[b, j]:
                    drafts[b, j] = am[b, j - 1]
        seq_h = kv_h + ql_h
        ref = oracle.greedy_accept(logits, drafts, q_lens=ql_h,
                                   seq_lens=seq_h)
        prep = oracle.prepare_next_block(
            policy, q_max, ql_h, ref["accept_len"], ref["next_token"],
            ref["new_seq_lens"], state_h, pt, page_size=ps,
            num_pages=B * max_pages, **pol_kw)
        acc, nxt, _, new = sv.greedy_accept_commit(
            d(logits), d(drafts), ql_d, kv_d + ql_d)
        out = sv.prepare_next_block(pol, ql_d, acc, nxt, new, state_d, pt_d,
                                    page_size=ps, num_pages=B * max_pages)
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy(), ref["accept_len"])
        assert np.array_equal(new.cpu().numpy(), ref["new_seq_lens"])
        for k in ("next_q_lens", "next_seq_lens", "block_ids", "positions",
                  "cache_loc"):
            assert np.array_equal(out[k].cpu().numpy(), prep[k]), (step, k)
        assert np.array_equal(state_d.cpu().numpy(), prep["state"])
        state_h, ql_h, kv_h = prep["state"], prep["next_q_lens"], \
            ref["new_seq_lens"]
        ql_d, kv_d = out["next_q_lens"], new
