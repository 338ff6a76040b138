"""A verify step (attention + greedy accept) captured in a CUDA graph
replays to the same results as eager calls: the library only enqueues
kernels on the caller's stream and derives its work plan on the device."""
import pytest
import torch

import speculative_decoding_target_gb300 as sv
from speculative_decoding_target_gb300 import _native
from speculative_decoding_target_gb300 import workloads as wl
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("kv_dtype,ps", [("bf16", 16), ("fp8_e4m3", 64),
                                         ("bf16", 4)])
def test_graph_replay_matches_eager(kv_dtype, ps):
    ensure_built()
    inp = wl.make_attention_inputs(
        batch=3, q_len=8, num_q_heads=24, num_kv_heads=4, head_dim=256,
        page_size=ps, prefix_lens=[700, 3000, 65], kv_dtype=kv_dtype,
        seed=42, device=DEV)
    acc_in = wl.make_accept_inputs(batch=3, q_len=8, vocab=50_000,
                                   accept_p=0.7, seed=42, device=DEV)
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"])
    ws = sv.alloc_workspace(sv.verify_workspace_size(desc), DEV)
    aws = sv.alloc_workspace(sv.accept_workspace_size(24, 50_000), DEV)
    out = torch.empty_like(inp["q"])
    acc = torch.empty(3, dtype=torch.int32, device=DEV)
    nxt = torch.empty(3, dtype=torch.int32, device=DEV)
    toks = torch.empty((3, 8), dtype=torch.int32, device=DEV)
    stream = torch.cuda.Stream()

    def step():
        _native.verify_attention_into(
            desc, inp["q"], inp["k_pages"], inp["v_pages"], inp["k_scales"],
            inp["v_scales"], inp["page_table"], inp["seq_lens"], inp["scale"],
            out, ws, stream)
        _native.greedy_accept_into(acc_in["logits"], acc_in["draft_ids"], acc,
                                   nxt, toks, aws, stream)

    with torch.cuda.stream(stream):
        step()                      # eager (also primes per-device caches)
    stream.synchronize()
    ref = [t.clone() for t in (out, acc, nxt, toks)]
    for t in (out, acc, nxt, toks):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(2):
        for t in (out, acc, nxt, toks):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref[0].view(torch.int16))
        for a, b in zip((acc, nxt, toks), ref[1:]):
            assert torch.equal(a, b)
