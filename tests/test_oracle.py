"""Pins for the CPU float64 oracle (no GPU).

Each test checks the oracle against something other than itself: a library
routine (torch float64 scaled-dot-product attention, torch / numpy float
decoders, numpy argmax, scipy logsumexp), a closed form, an invariant the
pages fix, or a worked example the pages print (fixtures in tests/golden/).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_target_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoders --

def test_e4m3_decoder_every_byte_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    # fixed points of the OCP E4M3 format
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    assert ours[0x08] == 2.0 ** -6 and ours[0xB8] == -1.0


def test_fp16_decoder_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_fp16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_decoder_every_pattern_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(
        torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ------------------------------------------------------ attention helpers --

def _inputs(B=2, q_len=4, hq=6, hkv=2, d=64, ps=4, prefix=(9, 13),
            kv_dtype="bf16", seed=3, **kw):
    return wl.make_attention_inputs(batch=B, q_len=q_len, num_q_heads=hq,
                                    num_kv_heads=hkv, head_dim=d,
                                    page_size=ps, prefix_lens=list(prefix),
                                    kv_dtype=kv_dtype, seed=seed, **kw)


def _run_oracle(inp, **kw):
    bits = wl.to_numpy_bits
    fp8 = inp["k_scales"] is not None
    return oracle.verify_attention(
        bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
        inp["page_table"].numpy(), inp["seq_lens"].numpy(),
        num_kv_heads=inp["num_kv_heads"], scale=inp["scale"],
        k_scales=bits(inp["k_scales"]) if fp8 else None,
        v_scales=bits(inp["v_scales"]) if fp8 else None, **kw)


def _dense_kv_torch(inp, b, which):
    """Request b's logical K or V as float64 [Hkv, L, D], decoded by torch."""
    pages = inp[which + "_pages"]
    ps = pages.shape[2]
    L = int(inp["seq_lens"][b])
    n = math.ceil(L / ps)
    ids = inp["page_table"][b, :n].long()
    x = pages[ids]                                    # [n, Hkv, ps, D]
    if inp["k_scales"] is None:
        xf = x.to(torch.float64)
    else:
        sc = inp[which + "_scales"][ids].to(torch.float64)  # [n,Hkv,ps,D/64]
        xf = x.view(torch.float8_e4m3fn).to(torch.float64)
        xf = xf * sc.repeat_interleave(64, dim=-1)
    xf = xf.permute(1, 0, 2, 3).reshape(x.shape[1], n * ps, x.shape[3])
    return xf[:, :L]


def _sdpa_reference(inp):
    """torch float64 scaled_dot_product_attention per request, with GQA heads
    expanded and the verify block's causal-offset mask."""
    q = inp["q"].to(torch.float64)                    # [B, q, Hq, D]
    B, q_len, hq, d = q.shape
    hkv = inp["num_kv_heads"]
    outs = []
    for b in range(B):
        L = int(inp["seq_lens"][b])
        k = _dense_kv_torch(inp, b, "k").repeat_interleave(hq // hkv, dim=0)
        v = _dense_kv_torch(inp, b, "v").repeat_interleave(hq // hkv, dim=0)
        i = torch.arange(q_len).unsqueeze(1)
        t = torch.arange(L).unsqueeze(0)
        mask = t < (L - q_len + i + 1)                # [q, L] True = attend
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].transpose(0, 1), k, v, attn_mask=mask, scale=inp["scale"])
        outs.append(o.transpose(0, 1))                # [q, Hq, D]
    return torch.stack(outs).reshape(-1, d).numpy()


# -------------------------------------------------------- attention pins --

@pytest.mark.parametrize("kv_dtype,d,ps,q_len,hq,hkv,prefix", [
    ("bf16", 8, 4, 1, 4, 2, (0, 5)),
    ("bf16", 64, 4, 4, 6, 2, (9, 13)),
    ("bf16", 256, 16, 8, 24, 4, (40, 17)),
    ("bf16", 256, 16, 16, 12, 2, (70, 1)),
    ("fp8_e4m3", 64, 4, 3, 6, 3, (11, 2)),
    ("fp8_e4m3", 256, 16, 8, 24, 4, (33, 64)),
])
def test_oracle_matches_torch_sdpa(kv_dtype, d, ps, q_len, hq, hkv, prefix):
    inp = _inputs(B=len(prefix), q_len=q_len, hq=hq, hkv=hkv, d=d, ps=ps,
                  prefix=prefix, kv_dtype=kv_dtype, seed=11 + d + q_len)
    ours = _run_oracle(inp)
    ref = _sdpa_reference(inp)
    assert np.all(np.isfinite(ours))
    np.testing.assert_allclose(ours, ref, rtol=1e-11, atol=1e-12)


def test_lse_matches_scipy_logsumexp():
    from scipy.special import logsumexp
    inp = _inputs(B=1, q_len=3, hq=4, hkv=2, d=64, ps=4, prefix=(10,))
    _, lse = _run_oracle(inp, return_lse=True)
    q = inp["q"].to(torch.float64)[0]                 # [q, Hq, D]
    k = _dense_kv_torch(inp, 0, "k")
    L = int(inp["seq_lens"][0])
    for i in range(3):
        for h in range(4):
            s = (k[h // 2, :L - 3 + i + 1] @ q[i, h]) * inp["scale"]
            assert lse[i * 4 + h] == pytest.approx(logsumexp(s.numpy()),
                                                   rel=1e-13, abs=1e-13)


def _custom(q_rows, k_rows, v_rows, ps=4, scale=0.25):
    """A one-request, one-head, q_len-row problem from explicit float rows
    (exactly representable in bf16)."""
    q = torch.tensor(q_rows, dtype=torch.float32)
    k = torch.tensor(k_rows, dtype=torch.float32)
    v = torch.tensor(v_rows, dtype=torch.float32)
    q_len, d = q.shape
    L = k.shape[0]
    n = math.ceil(L / ps)
    kp = torch.zeros((n, 1, ps, d))
    vp = torch.zeros((n, 1, ps, d))
    kp.view(-1, d)[:L] = k
    vp.view(-1, d)[:L] = v
    return {"q": q.view(1, q_len, 1, d).to(torch.bfloat16),
            "k_pages": kp.to(torch.bfloat16), "v_pages": vp.to(torch.bfloat16),
            "k_scales": None, "v_scales": None,
            "page_table": torch.arange(n, dtype=torch.int32).view(1, n),
            "seq_lens": torch.tensor([L], dtype=torch.int32),
            "scale": scale, "num_kv_heads": 1}


def test_identical_keys_return_mean_of_v():
    rng = np.random.default_rng(0)
    L, d = 23, 8
    k_row = [0.5, -1.0, 2.0, 0.25, 1.0, -0.5, 0.75, 3.0]
    v = np.round(rng.normal(size=(L, d)) * 8) / 8
    q = np.round(rng.normal(size=(2, d)) * 4) / 4
    out = _run_oracle(_custom(q, [k_row] * L, v))
    # row i sees the first L-2+i+1 keys; all weights are equal
    for i in range(2):
        n = L - 2 + i + 1
        np.testing.assert_allclose(out[i], v[:n].mean(axis=0), rtol=0,
                                   atol=1e-14)


def test_dominant_key_returns_its_value():
    L, d = 17, 8
    k = np.zeros((L, d))
    k[5, 0] = 64.0
    q = np.zeros((1, d))
    q[0, 0] = 8.0                      # score 512 * 0.25 = 128 vs 0
    v = np.arange(L * d, dtype=np.float64).reshape(L, d) / 4
    out = _run_oracle(_custom(q, k, v))
    np.testing.assert_allclose(out[0], v[5], rtol=0, atol=1e-12)


@pytest.mark.parametrize("x", [0.0, 0.75, -2.5, 6.0])
def test_two_keys_give_sigmoid_weights(x):
    # one-hot V rows recover the softmax weights: w1 = 1 / (1 + e^-x)
    d = 4
    q = [[1.0, 0, 0, 0]]
    k = [[0.0, 0, 0, 0], [x * 4, 0, 0, 0]]   # scale 0.25 -> scores 0, x
    v = [[1.0, 0, 0, 0], [0, 1.0, 0, 0]]
    out = _run_oracle(_custom(q, k, v))
    w1 = 1.0 / (1.0 + math.exp(-x))
    assert out[0, 1] == pytest.approx(w1, rel=1e-14, abs=1e-15)
    assert out[0, 0] == pytest.approx(1.0 - w1, rel=1e-13, abs=1e-15)


def test_q1_block_equals_decode_and_rows_equal_q1_calls():
    """Row i of a q-block equals a q_len=1 call whose cache holds the prefix
    plus drafts 1..i (one call per position with its own cache length)."""
    inp = _inputs(B=2, q_len=5, hq=6, hkv=2, d=64, ps=4, prefix=(9, 13))
    full = _run_oracle(inp).reshape(2, 5, 6, 64)
    for b in range(2):
        P = int(inp["seq_lens"][b]) - 5
        for i in range(5):
            one = dict(inp)
            one["q"] = inp["q"][b:b + 1, i:i + 1].contiguous()
            one["page_table"] = inp["page_table"][b:b + 1].contiguous()
            one["seq_lens"] = torch.tensor([P + i + 1], dtype=torch.int32)
            o1 = _run_oracle(one).reshape(6, 64)
            assert np.array_equal(o1, full[b, i])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_split_merge_equals_unsplit(kv_dtype):
    inp = _inputs(B=1, q_len=4, hq=4, hkv=2, d=64, ps=4, prefix=(37,),
                  kv_dtype=kv_dtype, seed=5)
    full = _run_oracle(inp)
    L = int(inp["seq_lens"][0])
    rng = np.random.default_rng(1)
    for _ in range(4):
        cuts = sorted(rng.choice(np.arange(1, L), size=3, replace=False))
        bounds = [0] + list(cuts) + [L]
        parts = [_run_oracle(inp, key_begin=lo, key_end=hi, return_lse=True)
                 for lo, hi in zip(bounds[:-1], bounds[1:])]
        for r in range(full.shape[0]):
            lse = np.array([p[1][r] for p in parts])
            o = np.stack([p[0][r] for p in parts])
            merged, _ = oracle.lse_merge(lse, o)
            np.testing.assert_allclose(merged, full[r], rtol=1e-12,
                                       atol=1e-13)


def test_merge_closed_forms():
    o = np.array([[1.0, 2.0], [3.0, 6.0]])
    out, lse = oracle.lse_merge([0.5, 0.5], o)   # equal weights -> average
    np.testing.assert_allclose(out, [2.0, 4.0], rtol=1e-15)
    assert lse == pytest.approx(0.5 + math.log(2.0), rel=1e-15)
    out, lse = oracle.lse_merge([-math.inf, 1.25], o)  # empty part ignored
    np.testing.assert_allclose(out, [3.0, 6.0], rtol=1e-15)
    assert lse == 1.25
    out, lse = oracle.lse_merge([-math.inf, -math.inf], o)
    assert np.all(out == 0) and lse == -math.inf


def test_permuted_pool_and_poison_change_nothing():
    a = _inputs(B=2, q_len=4, hq=6, hkv=2, d=64, ps=4, prefix=(9, 14),
                shuffle=False, poison=False, spare_pages=0)
    # same logical content through a permuted pool with NaN-poisoned slots
    npg = a["k_pages"].shape[0]
    perm = torch.randperm(npg + 3, generator=torch.Generator().manual_seed(4))
    b = dict(a)
    for name in ("k_pages", "v_pages"):
        src = a[name]
        dst = torch.full((npg + 3,) + tuple(src.shape[1:]), float("nan"),
                         dtype=src.dtype)
        dst[perm[:npg]] = src
        b[name] = dst
    pt = a["page_table"].clone()
    valid = pt >= 0
    pt[valid] = perm[pt[valid].long()].to(torch.int32)
    b["page_table"] = pt
    for bb in range(2):       # poison the unused tail slots of the last page
        L = int(a["seq_lens"][bb])
        last = (L - 1) // 4
        for name in ("k_pages", "v_pages"):
            b[name][int(pt[bb, last]), :, L - last * 4:] = float("nan")
    oa, ob = _run_oracle(a), _run_oracle(b)
    assert np.all(np.isfinite(ob))
    assert np.array_equal(oa, ob)


def test_bad_page_id_is_reported_not_read():
    inp = _inputs(B=1, q_len=2, hq=2, hkv=1, d=64, ps=4, prefix=(6,))
    inp["page_table"][0, 1] = 10_000
    with pytest.raises(ValueError):
        _run_oracle(inp)


# ---------------------------------------------------------- accept pins --

def _accept_from_argmax(boundary, drafts, argmax_rows, vocab=20000):
    """Logits whose row argmaxes are the given ids (one-hot at 1.0)."""
    q_len = len(drafts) + 1
    assert len(argmax_rows) >= q_len
    logits = np.zeros((q_len, vocab), np.float32)
    for j in range(q_len):
        logits[j, argmax_rows[j]] = 1.0
    d = np.array([[boundary] + list(drafts)], np.int32)
    return oracle.greedy_accept(logits, d)


def test_accept_worked_examples_from_pages():
    with open(os.path.join(GOLDEN, "accept_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        rows = list(c["target_argmax_rows"])
        rows = rows + [rows[-1]] * (len(c["drafts"]) + 1 - len(rows))
        r = _accept_from_argmax(c["boundary"], c["drafts"], rows)
        assert int(r["accept_len"][0]) == c["expect_accept_len"], c["name"]
        assert int(r["next_token"][0]) == c["expect_next_token"], c["name"]
        if "expect_committed" in c:
            a = c["expect_accept_len"]
            assert r["out_tokens"][0, :a + 1].tolist() == c["expect_committed"]
            assert np.all(r["out_tokens"][0, a + 1:] == -1)


def test_all_accept_and_first_mismatch():
    rows = [5, 6, 7, 8, 9]
    r = _accept_from_argmax(1, [5, 6, 7, 8], rows)
    assert r["accept_len"][0] == 4 and r["next_token"][0] == 9   # k+1 tokens
    assert r["out_tokens"][0].tolist() == [5, 6, 7, 8, 9]
    r = _accept_from_argmax(1, [4, 6, 7, 8], rows)
    assert r["accept_len"][0] == 0 and r["next_token"][0] == 5   # 1 token
    assert r["out_tokens"][0].tolist() == [5, -1, -1, -1, -1]
    r = _accept_from_argmax(1, [], [3])                            # q_len = 1
    assert r["accept_len"][0] == 0 and r["next_token"][0] == 3


def test_argmax_exhaustive_ties_match_numpy():
    vals = np.array([-1.0, -0.0, 0.0, 1.0, np.nan], np.float32)
    idx = np.stack(np.meshgrid(*[np.arange(5)] * 4, indexing="ij"), -1)
    logits = vals[idx.reshape(-1, 4)]                 # 625 rows, vocab 4
    drafts = np.zeros((logits.shape[0], 1), np.int32)
    r = oracle.greedy_accept(logits, drafts)
    assert np.array_equal(r["argmax"], np.argmax(logits, axis=1))
    assert np.array_equal(r["next_token"], np.argmax(logits, axis=1))


def test_speculative_commit_stream_equals_serial_greedy():
    """Committing d1..da plus the target token at the first disagreement
    reproduces serial greedy decoding token for token."""
    V, rng = 12, np.random.default_rng(7)
    table = rng.integers(0, V, size=(V, V))

    def target_next(ctx):                 # a deterministic toy target
        return int(table[ctx[-2] if len(ctx) > 1 else 0, ctx[-1]])

    serial = [3]
    while len(serial) < 200:
        serial.append(target_next(serial))

    stream = [3]
    steps = 0
    while len(stream) < 200:
        q_len = int(rng.integers(1, 9))
        drafts, ctx = [], list(stream)
        for _ in range(q_len - 1):        # a drafter that is right ~60%
            t = target_next(ctx)
            d = t if rng.random() < 0.6 else int(rng.integers(0, V))
            drafts.append(d)
            ctx.append(d)
        logits = rng.normal(size=(q_len, V)).astype(np.float32)
        ctx = list(stream)
        for j in range(q_len):            # row j scores the token after
            logits[j, target_next(ctx)] = 50.0      # block position j
            if j < q_len - 1:
                ctx.append(drafts[j])
        r = oracle.greedy_accept(logits, np.array([[stream[-1]] + drafts],
                                                  np.int32))
        a = int(r["accept_len"][0])
        committed = r["out_tokens"][0, :a + 1].tolist()
        assert committed[-1] == int(r["next_token"][0])
        stream.extend(committed)
        steps += 1
    assert stream[:200] == serial
    assert steps < 199                    # some drafts were accepted


def test_survival_rates_sum_to_mean_accept():
    with open(os.path.join(GOLDEN, "survival_rates.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:   # the pages' own numbers obey the identity
        assert sum(c["survival_percent"]) / 100 == pytest.approx(
            c["mean_accepted"], abs=1e-4)
    # and so do the oracle's accept lengths on planted drafts, whose mean is
    # sum_j p^j for independent per-position planting
    B, q_len, p = 2048, 8, 0.5
    inp = wl.make_accept_inputs(batch=B, q_len=q_len, vocab=64, accept_p=p,
                                seed=9)
    r = oracle.greedy_accept(inp["logits"].numpy(), inp["draft_ids"].numpy())
    a = r["accept_len"]
    surv = [(a >= j).mean() for j in range(1, q_len)]
    assert sum(surv) == pytest.approx(a.mean(), abs=1e-12)
    assert a.mean() == pytest.approx(sum(p ** j for j in range(1, q_len)),
                                     abs=0.08)


def test_kv_byte_formula_matches_pages():
    with open(os.path.join(GOLDEN, "kv_bytes.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = c["layers"] * wl.kv_bytes(
            [c["tokens"]], c["kv_heads"], c["head_dim"], c["kv_dtype"],
            include_scales=not c.get("exclude_scales", False))
        assert got == c["expect_bytes"], c["name"]
