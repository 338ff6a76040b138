"""GPU DFlash2 candidate selection (through the C ABI) against the oracle:
candidate ids and logits bit for bit, transition tables within float32
accumulation error, and the chosen chains equal wherever the oracle's
smallest decision gap exceeds what float32 rounding can move."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"
GAP = 1e-3         # chains may differ only where a decision was this close


def _case(B, P, V, R, D, seed, scale=0.3, ties=False):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn((B, P - 1, V), generator=g) * 2
    if ties:      # repeated maxima and -inf stretches exercise the order
        logits[:, :, 100:200] = 7.0
        logits[0, 0, : V // 2] = float("-inf")
    return dict(
        cand_logits=logits,
        boundary=torch.randint(0, V, (B,), generator=g, dtype=torch.int32),
        hidden=torch.randn((B, P - 1, D), generator=g).to(torch.bfloat16),
        w_h=(torch.randn((R, D), generator=g) / D ** 0.5).to(torch.bfloat16),
        code_a=(torch.randn((V, R), generator=g) * scale).to(torch.bfloat16),
        code_b=(torch.randn((V, R), generator=g) * scale).to(torch.bfloat16))


def _compare(inp, top, mode):
    ensure_built()
    dev = {k: v.to(DEV) for k, v in inp.items()}
    got = sv.dflash2_select(dev["cand_logits"], dev["boundary"], dev["hidden"],
                            dev["w_h"], dev["code_a"], dev["code_b"], top=top,
                            mode=mode)
    torch.cuda.synchronize()
    bits = wl.to_numpy_bits
    ref = oracle.dflash2_select(
        inp["cand_logits"].numpy(), inp["boundary"].numpy(),
        bits(inp["hidden"]), bits(inp["w_h"]), bits(inp["code_a"]),
        bits(inp["code_b"]), top=top, mode=mode)
    assert np.array_equal(got["cand_ids"].cpu().numpy(), ref["cand_ids"])
    assert np.array_equal(got["cand_logit"].cpu().numpy().astype(np.float64),
                          ref["cand_logit"])
    tr = got["trans"].cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref["trans"])
    assert np.array_equal(np.isfinite(tr), fin)
    err = np.abs(tr[fin] - ref["trans"][fin])
    assert err.max() <= 1e-4 + 1e-5 * np.abs(ref["trans"][fin]).max(), \
        err.max()
    d = got["draft_ids"].cpu().numpy()
    assert np.array_equal(d[:, 0], inp["boundary"].numpy())
    same = (d == ref["draft_ids"]).all(1)
    flips = np.flatnonzero(~same)
    assert np.all(ref["margin"][flips] < GAP), (flips, ref["margin"][flips])
    assert len(flips) <= max(1, len(same) // 20)
    return ref


@pytest.mark.parametrize("mode", ["greedy", "map"])
@pytest.mark.parametrize("B,P,V,R,D,top", [
    (4, 8, 30000, 64, 256, 16), (3, 5, 8192, 256, 512, 16),
    (2, 16, 9000, 32, 128, 8), (6, 2, 20001, 16, 64, 4),
    (5, 8, 1000, 8, 16, 1)])
def test_matches_oracle(B, P, V, R, D, top, mode):
    _compare(_case(B, P, V, R, D, seed=B * P + V), top, mode)


def test_ties_and_infinities():
    _compare(_case(3, 6, 5000, 32, 64, seed=9, ties=True), 16, "greedy")


def test_production_shape():
    # 8 requests x 8 positions, top 16 of 248,320, rank 256, hidden 5,120
    ref = _compare(_case(8, 8, 248320, 256, 5120, seed=1), 16, "greedy")
    assert ref["draft_ids"].shape == (8, 8)
    _compare(_case(8, 8, 248320, 256, 5120, seed=2), 16, "map")


def test_zero_codebooks_give_the_argmax_chain():
    inp = _case(4, 8, 12000, 32, 64, seed=3)
    inp["code_a"].zero_()
    ensure_built()
    dev = {k: v.to(DEV) for k, v in inp.items()}
    for mode in ("greedy", "map"):
        got = sv.dflash2_select(dev["cand_logits"], dev["boundary"],
                                dev["hidden"], dev["w_h"], dev["code_a"],
                                dev["code_b"], mode=mode)
        am = inp["cand_logits"].argmax(dim=2).to(torch.int32)
        assert torch.equal(got["draft_ids"][:, 1:].cpu(), am)
