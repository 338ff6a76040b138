"""GPU greedy acceptance (through the C ABI) against the oracle: bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run_both(logits: torch.Tensor, drafts: torch.Tensor):
    ensure_built()
    import speculative_decoding_target_gb300 as sv
    acc, nxt, toks = sv.greedy_accept(logits, drafts)
    torch.cuda.synchronize()
    ref = oracle.greedy_accept(logits.cpu().numpy(), drafts.cpu().numpy())
    assert np.array_equal(acc.cpu().numpy(), ref["accept_len"])
    assert np.array_equal(nxt.cpu().numpy(), ref["next_token"])
    assert np.array_equal(toks.cpu().numpy(), ref["out_tokens"])
    return ref


@pytest.mark.parametrize("B,q_len,vocab,p", [
    (1, 8, 248320, 0.5), (3, 16, 100003, 0.7), (5, 1, 4096, 0.5),
    (2, 5, 8191, 0.9), (4, 8, 8193, 1.0), (2, 8, 7, 0.5), (1, 2, 1, 1.0),
    (6, 8, 1023, 0.6), (6, 8, 1024, 0.6), (6, 8, 1025, 0.6), (9, 3, 2052, 0.8),
])
def test_random_planted(B, q_len, vocab, p):
    inp = wl.make_accept_inputs(batch=B, q_len=q_len, vocab=vocab,
                                accept_p=p, seed=B * 100 + q_len, device=DEV)
    _run_both(inp["logits"], inp["draft_ids"])


@pytest.mark.parametrize("V", [3 * 8192 + 17, 3 * 8192 + 16])
def test_ties_zeros_and_nan(V):
    # V % 4 == 0 with aligned rows takes the 16-byte load path, otherwise
    # the scalar one
    q_len = 8
    g = torch.Generator().manual_seed(0)
    base = torch.randn((q_len * 4, V), generator=g)
    # row 0: the maximum repeated in several chunks -> lowest index
    base[0, [20000, 9000, 24000, 5]] = 50.0
    # row 1: every entry equal -> index 0
    base[1] = 1.5
    # row 2: only -0.0 and +0.0 -> index 0 (they compare equal)
    base[2] = 0.0
    base[2, ::2] = -0.0
    base[2, 0] = -0.0
    # row 3: NaNs in two chunks -> the first NaN wins
    base[3, 17000] = float("nan")
    base[3, 8200] = float("nan")
    # row 4: -inf everywhere except one finite value near the end
    base[4] = float("-inf")
    base[4, V - 1] = -1e30
    # row 5: the maximum at the last index
    base[5, V - 1] = 1e9
    logits = base.to(DEV)
    am = [0, 0, 0, 8200, V - 1, V - 1]
    drafts = torch.zeros((4, q_len), dtype=torch.int32)
    drafts[0, 1:] = torch.tensor([5, 0, 0, 8200, V - 1, V - 1, 3])
    ref = _run_both(logits, drafts.to(DEV))
    assert ref["argmax"][:6].tolist() == [5] + am[1:]


def test_unaligned_logits_take_the_scalar_path():
    inp = wl.make_accept_inputs(batch=3, q_len=4, vocab=50000, accept_p=0.8,
                                seed=1, device=DEV)
    # a view starting one float in: rows no longer 16-byte aligned
    big = torch.empty(inp["logits"].numel() + 1, device=DEV)
    big[1:] = inp["logits"].reshape(-1)
    view = big[1:].view(12, 50000)
    _run_both(view, inp["draft_ids"])


def test_worked_examples_from_pages():
    with open(os.path.join(GOLDEN, "accept_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q_len = len(c["drafts"]) + 1
        rows = list(c["target_argmax_rows"])
        rows += [rows[-1]] * (q_len - len(rows))
        logits = torch.randn((q_len, 30000), generator=torch.Generator()
                             .manual_seed(2))
        for j in range(q_len):
            logits[j, rows[j]] = 100.0
        drafts = torch.tensor([[c["boundary"]] + c["drafts"]], dtype=torch.int32)
        ref = _run_both(logits.to(DEV), drafts.to(DEV))
        assert ref["accept_len"][0] == c["expect_accept_len"]
        assert ref["next_token"][0] == c["expect_next_token"]


@pytest.mark.parametrize("name", wl.WORKLOAD_ORDER)
def test_full_size_workloads(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_accept_inputs(batch=w.batch, q_len=w.q_len, vocab=w.vocab,
                                accept_p=w.accept_p, seed=w.seed, device=DEV)
    ref = _run_both(inp["logits"], inp["draft_ids"])
    # survival rates sum to the mean accepted length
    a = ref["accept_len"]
    assert sum((a >= j).mean() for j in range(1, w.q_len)) == \
        pytest.approx(a.mean(), abs=1e-12)


def test_row_limit():
    # batch * q_len up to the 65,535-row limit of the argmax grid
    inp = wl.make_accept_inputs(batch=4095, q_len=16, vocab=33, accept_p=0.9,
                                seed=4095, device=DEV)
    _run_both(inp["logits"], inp["draft_ids"])
