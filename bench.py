#!/usr/bin/env python3
"""Benchmark of the target-verify step: paged GQA verify attention followed
by greedy acceptance, on seeded synthetic inputs, through the C ABI.

One step = spec_verify_attention (split-KV kernel + LSE merge) over every
request's verify block, then spec_greedy_accept over the block's logits.
Default workload: batch 8, q_len 8, 24/4 heads, head_dim 256, 32,768-token
prefixes in 64-token pages of a permuted pool, bf16 KV; logits
[64 x 248,320] fp32 with drafts planted at p = 0.6.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica of the workload on its own GPU (the step has no cross-GPU exchange),
timing is the max over ranks, and value counts the steps of all ranks.

--impl reference times the CPU float64 oracle on the host cores instead
(rank 0 only), on a bounded sample of rows per step, extrapolated to the
whole workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_target_gb300 import workloads as wl  # noqa: E402

METRIC = ("verify steps/s and KV-read GB/s (fraction of GB300 HBM peak) at "
          "1 GPU")
UNIT = "steps/s"
DEFAULT_WORKLOAD = "b8_q8_p32k"
KERNEL_LAUNCHES_PER_STEP = 3   # split, merge, argmax (its last CTA per request finalises)

# DRAM traffic of one launch of the dominant kernel (the split-KV attention
# kernel), dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture
# (profiles/verify_split_*.md), keyed by workload and valid only while that
# kernel's sources still hash to the recorded value.
NCU_TRAFFIC = {
    "b8_q8_p32k": {"kernel": "tc", "source_hash": "82f85a10d3d072aa",
                   "bytes_per_launch": 1077388032 + 4466944},
    # captured on the smaller FP8 case b8_q8_p16k_fp8 (276.95 MB
    # algorithmic: 279.21 MB read + 4.59 MB written) and scaled to a full
    # launch by the algorithmic bytes, which the traffic follows
    "b32_q8_p1k128k_fp8": {"kernel": "fp8t", "source_hash": "70ac74e863844017",
                           "per_algorithmic_byte": (279210496 + 4592896)
                           / (8 * 16392 * 4 * 528)},
}
NCU_TRAFFIC["b8_q8_p16k_fp8"] = NCU_TRAFFIC["b32_q8_p1k128k_fp8"]

# Sources of each split kernel: bf16 KV and FP8 blocks of more than 64 rows
# per KV head take the tcgen05 kernel with Q in tensor memory; FP8 blocks of
# at most 64 rows take the kernel with K and V^T in tensor memory.
KERNEL_SOURCES = {
    "tc": ("verify_attention_tc.cu", "common.cuh", "tc_ptx.cuh"),
    "fp8t": ("verify_attention_fp8t.cu", "tmem_io.cuh", "common.cuh",
             "tc_ptx.cuh"),
}


def split_kernel_of(w) -> str:
    rows = w.q_len * (w.num_q_heads // w.num_kv_heads)
    return "fp8t" if w.kv_dtype != "bf16" and rows <= 64 else "tc"


def kernel_source_hash(kind: str = "tc") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_target_gb300", "csrc")
    for fn in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        self.ident = ident

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident,
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks of the default process group (the value
    itself when there is no group).  Timing uses the slowest rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or \
            dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, elapsed_ms: float) -> float:
    """Steps of the whole job per second: every rank runs `steps` steps of
    its own replica, and the job takes as long as its slowest rank."""
    return world * steps / (elapsed_ms / 1e3)


def algorithmic_bytes(w: wl.VerifyWorkload, seq_lens):
    kv = wl.kv_bytes(seq_lens, w.num_kv_heads, w.head_dim, w.kv_dtype)
    logits = w.batch * w.q_len * w.vocab * 4
    return kv, logits


# ----------------------------------------------------------------- GPU arm --

def run_gpu(args, w: wl.VerifyWorkload):
    import speculative_decoding_target_gb300 as sv
    from speculative_decoding_target_gb300 import _native

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sv.load()

    inp = wl.workload_inputs(w, device=dev)
    seq_lens = inp["seq_lens"].tolist()
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"])
    attn_ws = sv.alloc_workspace(sv.verify_workspace_size(desc), dev)
    rows = w.batch * w.q_len
    acc_ws = sv.alloc_workspace(sv.accept_workspace_size(rows, w.vocab), dev)
    out = torch.empty_like(inp["q"])
    acc = torch.empty(w.batch, dtype=torch.int32, device=dev)
    nxt = torch.empty(w.batch, dtype=torch.int32, device=dev)
    toks = torch.empty((w.batch, w.q_len), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev_a=None, ev_b=None):
        if ev_a is not None:
            ev_a.record(stream)
        _native.verify_attention_into(
            desc, inp["q"], inp["k_pages"], inp["v_pages"], inp["k_scales"],
            inp["v_scales"], inp["page_table"], inp["seq_lens"], inp["scale"],
            out, attn_ws, stream)
        if ev_b is not None:
            ev_b.record(stream)
        _native.greedy_accept_into(inp["logits"], inp["draft_ids"], acc, nxt,
                                   toks, acc_ws, stream)

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if args.graph:
        # one CUDA graph per C-ABI call, replayed in the timed loop: the
        # same kernels without the per-call host overhead
        eager_step = step
        g_attn, g_acc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g_attn, stream=side):
                _native.verify_attention_into(
                    desc, inp["q"], inp["k_pages"], inp["v_pages"],
                    inp["k_scales"], inp["v_scales"], inp["page_table"],
                    inp["seq_lens"], inp["scale"], out, attn_ws, side)
            with torch.cuda.graph(g_acc, stream=side):
                _native.greedy_accept_into(inp["logits"], inp["draft_ids"],
                                           acc, nxt, toks, acc_ws, side)
        torch.cuda.synchronize(dev)

        def step(ev_a=None, ev_b=None):
            if ev_a is not None:
                ev_a.record(stream)
            g_attn.replay()
            if ev_b is not None:
                ev_b.record(stream)
            g_acc.replay()

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        del eager_step

    evs = [(torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for k in range(args.steps):
        step(*evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    attn_ms = [a.elapsed_time(b) for a, b in evs]
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and reads its results back
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, w, inp, desc, attn_ws, acc_ws, out, stream,
                          dev, ws_n, barrier)

    kv_b, logit_b = algorithmic_bytes(w, seq_lens)
    attn_avg_s = statistics.mean(attn_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved = kv_b / attn_avg_s / 1e9
    src_hash = kernel_source_hash(split_kernel_of(w))
    traffic = None
    rec = NCU_TRAFFIC.get(w.name)
    if rec and rec.get("source_hash") == src_hash:
        traffic = rec.get("bytes_per_launch")
        if traffic is None:
            traffic = int(rec["per_algorithmic_byte"] * kv_b)
    result = {
        "metric": METRIC,
        "value": round(job_throughput(ws_n, args.steps, elapsed_ms), 3),
        "unit": UNIT,
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == "bf16" else "fp8_e4m3",
        "data": "synthetic (seeded; random bf16 Q/K/V ~N(0,1), fp32 logits "
                "~N(0,4), planted drafts)",
        "config": {
            "workload": w.name, "batch": w.batch, "q_len": w.q_len,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "prefix": w.prefix or "U[1024,131072]",
            "page_size": w.page_size, "kv_dtype": w.kv_dtype,
            "vocab": w.vocab, "accept_p": w.accept_p,
            "kv_bytes_per_step": kv_b, "logits_bytes_per_step": logit_b,
            "l2": f"inputs larger than L2 ({(kv_b + logit_b) / 1e9:.3f} GB "
                  "read per step), no flush",
            "parallelism": f"replicas x{ws_n}",
            "cuda_graph": bool(args.graph),
        },
        "kv_read_gbs": round(achieved, 1),
        "roofline": {
            "kernel": "verify attention (split-KV kernel + LSE merge, one "
                      "C-ABI call)",
            "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": kv_b,
            "avg_launch_ms": round(attn_avg_s * 1e3, 5),
        },
        "gpu_launches": KERNEL_LAUNCHES_PER_STEP * args.steps,
        "kernel_source_hash": src_hash,
        "clocks": clk,
    }
    if e2e is not None:
        result["e2e"] = e2e
    if not args.no_append:
        result["kv_append"] = measure_kv_append(w, dev, args.steps,
                                                args.warmup)
    if not args.no_ragged:
        result["ragged"] = measure_ragged(w, inp, dev, args.steps,
                                          args.warmup, attn_avg_s)
    if not args.no_stochastic:
        result["stochastic"] = measure_stochastic(w, inp, dev, args.steps,
                                                  args.warmup, peak)
    if not args.no_select:
        result["dflash2_select"] = measure_select(w, dev, args.steps,
                                                  args.warmup, peak)
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        host_inp = {k: (v.cpu() if torch.is_tensor(v) else v)
                    for k, v in inp.items()}
        result["cpu_baseline"] = cpu_baseline(w, host_inp, args.cpu_seconds)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result, rank


# ------------------------------------------------------------- end to end --

def measure_e2e(args, w, inp, desc, attn_ws, acc_ws, out, stream, dev, ws_n,
                barrier):
    """The verify step through the public API with host buffers: every step
    copies its q, page table, seq_lens, logits and drafts in from pinned host
    memory and reads its out / accept / next / tokens back.  Two sets of
    device buffers let step k+1's copy-in (one stream) and step k-1's
    read-back (another) overlap step k's kernels; events keep each set's
    copy-in after the compute that last read it and its compute after the
    read-back of its previous result.  The KV pool stays resident: it is
    the cache state, not a per-step input."""
    from speculative_decoding_target_gb300 import _native
    keys = ("q", "page_table", "seq_lens", "logits", "draft_ids")
    # each direction is one contiguous staging buffer (tensors at 256-byte
    # offsets), so a step costs one host-to-device and one device-to-host
    # copy call whatever the number of tensors
    in_specs = [(k, inp[k].dtype, tuple(inp[k].shape)) for k in keys]
    out_specs = [("out", out.dtype, tuple(out.shape)),
                 ("acc", torch.int32, (w.batch,)),
                 ("nxt", torch.int32, (w.batch,)),
                 ("toks", torch.int32, (w.batch, w.q_len))]

    def packed(specs, device, pin):
        offs, n = [], 0
        for _, dt, shape in specs:
            offs.append(n)
            nb = torch.Size(shape).numel() * torch.empty((), dtype=dt).element_size()
            n += (nb + 255) // 256 * 256
        buf = torch.empty(n, dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = {}
        for (name, dt, shape), o in zip(specs, offs):
            nb = torch.Size(shape).numel() * torch.empty((), dtype=dt).element_size()
            views[name] = buf[o:o + nb].view(dt).view(shape)
        return buf, views

    h_in_buf, host = packed(in_specs, "cpu", True)
    for k in keys:
        host[k].copy_(inp[k].cpu())
    dev_in_bufs, dev_in = zip(*[packed(in_specs, dev, False) for _ in range(2)])
    dev_out_bufs, dev_out = zip(*[packed(out_specs, dev, False)
                                  for _ in range(2)])
    h_out_bufs, h_out = zip(*[packed(out_specs, "cpu", True) for _ in range(2)])
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    s_in, s_back = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    copied = [ev(), ev()]
    computed = [ev(), ev()]
    read = [ev(), ev()]
    used = [False, False]

    def copy_in(k):
        b = k & 1
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(computed[b])  # the set's last reader is done
            dev_in_bufs[b].copy_(h_in_buf, non_blocking=True)
            copied[b].record(s_in)

    def compute(k):
        b = k & 1
        stream.wait_event(copied[b])
        if used[b]:
            stream.wait_event(read[b])  # the set's last result was read back
        d, o = dev_in[b], dev_out[b]
        _native.verify_attention_into(
            desc, d["q"], inp["k_pages"], inp["v_pages"], inp["k_scales"],
            inp["v_scales"], d["page_table"], d["seq_lens"], inp["scale"],
            o["out"], attn_ws, stream)
        _native.greedy_accept_into(d["logits"], d["draft_ids"], o["acc"],
                                   o["nxt"], o["toks"], acc_ws, stream)
        computed[b].record(stream)
        used[b] = True

    def read_back(k):
        b = k & 1
        with torch.cuda.stream(s_back):
            s_back.wait_event(computed[b])
            h_out_bufs[b].copy_(dev_out_bufs[b], non_blocking=True)
            read[b].record(s_back)

    def run(n, start_ev=None):
        if start_ev is not None:
            s_in.wait_event(start_ev)
        copy_in(0)
        for k in range(n):
            compute(k)
            if k + 1 < n:
                copy_in(k + 1)  # overlaps compute(k)
            read_back(k)
        stream.wait_event(read[(n - 1) & 1])

    run(args.warmup)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(args.steps, e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    return {"value": round(job_throughput(ws_n, args.steps, e_ms), 3),
            "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "note": "KV pool resident in HBM (it is the cache state); every "
                    "step copies its q, page table, seq_lens, logits and "
                    "drafts in from pinned host memory and its out / "
                    "accept / next / tokens back (one staging buffer per "
                    "direction), double-buffered so that copies overlap "
                    "the previous step's kernels"}


# ------------------------------------------------------ block KV append --

def append_bytes(w: wl.VerifyWorkload) -> int:
    """Algorithmic bytes of one append: the block's bf16 K and V read, the
    pool rows written (E4M3 bytes + fp16 scales for FP8), positions and
    cache locations written."""
    rows = w.batch * w.q_len * w.num_kv_heads
    read = 2 * rows * w.head_dim * 2
    if w.kv_dtype == "bf16":
        write = 2 * rows * w.head_dim * 2
    else:
        write = 2 * rows * (w.head_dim + 2 * (w.head_dim // 64))
    return read + write + w.batch * w.q_len * (4 + 8)


def measure_kv_append(w: wl.VerifyWorkload, dev, iters: int, warmup: int):
    """Time spec_kv_append on the workload's block shape.  Its work depends
    on (batch, q_len, KV heads, head_dim, page size, KV dtype) only, so the
    pool here holds one page per request beyond the block."""
    import speculative_decoding_target_gb300 as sv
    inp = wl.make_attention_inputs(
        batch=w.batch, q_len=w.q_len, num_q_heads=w.num_q_heads,
        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        page_size=w.page_size, prefix_lens=[w.page_size] * w.batch,
        kv_dtype=w.kv_dtype, seed=w.seed, device=dev, poison=False)
    g = torch.Generator(device=dev).manual_seed(w.seed + 11)
    shape = (w.batch, w.q_len, w.num_kv_heads, w.head_dim)
    k_new = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    pos = torch.empty((w.batch, w.q_len), dtype=torch.int32, device=dev)
    loc = torch.empty((w.batch, w.q_len), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(st):
        sv.kv_append(k_new, v_new, inp["k_pages"], inp["v_pages"],
                     inp["page_table"], inp["seq_lens"],
                     k_scales=inp["k_scales"], v_scales=inp["v_scales"],
                     positions=pos, cache_loc=loc, stream=st)

    for _ in range(warmup):
        call(stream)
    torch.cuda.synchronize(dev)
    # device time: a CUDA graph of `iters` appends, replayed; eager calls
    # back to back would measure the host's submission rate instead
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(iters):
                call(side)
    torch.cuda.synchronize(dev)
    for _ in range(warmup):
        graph.replay()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    reps = 5
    a.record(stream)
    for _ in range(reps):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    us = a.elapsed_time(b) * 1e3 / (iters * reps)
    nbytes = append_bytes(w)
    return {"avg_us": round(us, 3), "algorithmic_bytes": nbytes,
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "launches": iters * reps,
            "note": f"{iters} spec_kv_append calls captured in one CUDA "
                    f"graph, replayed {reps} times; the block (<1% of L2) "
                    "stays warm in L2, so the figure is launch and latency "
                    "bound, not HBM bound"}


# ------------------------------------------------ per-request verify widths --

def measure_ragged(w: wl.VerifyWorkload, inp, dev, steps: int, warmup: int,
                   full_attn_s: float):
    """One verify step with per-request widths q_b ~ U[1, q_len] (seeded):
    attention over the padded block, accept with commit lengths (only the
    q_b logits rows of each request are read), and the next block's
    preparation under the EWMA width policy.  Timed per part with CUDA
    events over `steps` steps on the workload's resident inputs."""
    import speculative_decoding_target_gb300 as sv
    from speculative_decoding_target_gb300 import _native
    g = torch.Generator().manual_seed(w.seed + 21)
    ql_h = torch.randint(1, w.q_len + 1, (w.batch,), generator=g)
    ql = ql_h.to(torch.int32).to(dev)
    desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"],
                       q_lens=ql)
    attn_ws = sv.alloc_workspace(sv.verify_workspace_size(desc), dev)
    acc_ws = sv.alloc_workspace(
        sv.accept_workspace_size(w.batch * w.q_len, w.vocab), dev)
    out = torch.empty_like(inp["q"])
    i32 = dict(dtype=torch.int32, device=dev)
    acc, nxt, new = (torch.empty(w.batch, **i32) for _ in range(3))
    toks = torch.empty((w.batch, w.q_len), **i32)
    pol = sv.width_policy("ewma", w.q_len)
    state0 = torch.full((w.batch,), w.q_len - 1.0, device=dev)
    state = state0.clone()
    nq, nsl = torch.empty(w.batch, **i32), torch.empty(w.batch, **i32)
    bids, pos = (torch.empty((w.batch, w.q_len), **i32) for _ in range(2))
    loc = torch.empty((w.batch, w.q_len), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    num_pages = inp["k_pages"].shape[0]

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        _native.verify_attention_into(
            desc, inp["q"], inp["k_pages"], inp["v_pages"], inp["k_scales"],
            inp["v_scales"], inp["page_table"], inp["seq_lens"], inp["scale"],
            out, attn_ws, stream)
        if ev:
            ev[1].record(stream)
        sv.greedy_accept_commit_into(inp["logits"], inp["draft_ids"], ql,
                                     inp["seq_lens"], new, acc, nxt, toks,
                                     acc_ws, stream)
        if ev:
            ev[2].record(stream)
        sv.prepare_next_block_into(pol, ql, acc, nxt, new, state,
                                   inp["page_table"], w.page_size, num_pages,
                                   nq, nsl, bids, pos, loc, None, stream)
        if ev:
            ev[3].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
           for _ in range(steps)]
    for k in range(steps):
        step(evs[k])
    torch.cuda.synchronize(dev)
    part = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
            for j in range(3)]
    total = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
    rows = int(ql_h.sum())
    return {
        "value": round(1e3 / total, 3), "unit": UNIT,
        "widths": "q_b ~ U[1, q_len], seeded, the same every step; the "
                  "EWMA policy prepares the next block",
        "mean_width": round(rows / w.batch, 3),
        "attention_ms": round(part[0], 5),
        "attention_full_width_ms": round(full_attn_s * 1e3, 5),
        "accept_commit_ms": round(part[1], 5),
        "logits_bytes_read": rows * w.vocab * 4,
        "prepare_ms": round(part[2], 5),
        "gpu_launches": 4 * steps,
        "note": "attention streams the same KV whatever the widths (rows "
                "are free in the 128-row MMA tile); accept reads only the "
                "q_b logits rows of each request",
    }


# ------------------------------------------------------ stochastic verify --

def measure_stochastic(w: wl.VerifyWorkload, inp, dev, steps: int,
                       warmup: int, peak: float):
    """Rejection-sampling accept on the workload's logits: greedy drafts
    (no draft probabilities) and drafts with full draft distributions
    (B x (q_len - 1) x V fp32, the residual row read at a rejection).
    Temperature 1, seeded uniforms; CUDA events per call."""
    import speculative_decoding_target_gb300 as sv
    B, q, V = w.batch, w.q_len, w.vocab
    g = torch.Generator(device=dev).manual_seed(w.seed + 31)
    temp = torch.ones(B, device=dev)
    ua = torch.rand((B, max(q - 1, 1)), generator=g, device=dev)
    us = torch.rand(B, generator=g, device=dev)
    probs = torch.softmax(torch.randn((B, max(q - 1, 1), V), generator=g,
                                      device=dev), dim=-1)
    ws = sv.alloc_workspace(sv.stochastic_workspace_size(B, q, V), dev)
    i32 = dict(dtype=torch.int32, device=dev)
    acc, nxt = torch.empty(B, **i32), torch.empty(B, **i32)
    toks = torch.empty((B, q), **i32)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, dp in (("greedy_drafts", None), ("draft_probs", probs)):
        def call():
            sv.stochastic_accept_into(inp["logits"], inp["draft_ids"], dp,
                                      None, temp, ua, us, None, None, acc,
                                      nxt, toks, ws, stream)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        out[name + "_ms"] = round(ms, 5)
    logit_bytes = B * q * V * 4
    out.update({
        "logits_bytes": logit_bytes,
        "logits_gbs_greedy_drafts": round(
            logit_bytes / (out["greedy_drafts_ms"] * 1e-3) / 1e9, 1),
        "frac_of_peak_greedy_drafts": round(
            logit_bytes / (out["greedy_drafts_ms"] * 1e-3) / 1e9 / peak, 4),
        "gpu_launches": 3 * 2 * steps,
        "note": "three launches per call: one streaming pass over the logits "
                "(softmax statistics), per-chunk draw weights, the draw; "
                "temperature 1, seeded uniforms",
    })
    return out


# ------------------------------------------------------ DFlash2 selector --

SELECT_RANK, SELECT_HIDDEN, SELECT_TOP = 256, 5120, 16


def select_bytes(w: wl.VerifyWorkload) -> int:
    """Algorithmic bytes of one selection: the candidate logits of the
    drafted positions, the projection weights and hidden states, and the
    2 x K codebook rows gathered per position (bf16)."""
    rows = w.batch * (w.q_len - 1)
    return (rows * w.vocab * 4 + SELECT_RANK * SELECT_HIDDEN * 2 +
            rows * SELECT_HIDDEN * 2 + rows * 2 * SELECT_TOP * SELECT_RANK * 2)


def measure_select(w: wl.VerifyWorkload, dev, steps: int, warmup: int,
                   peak: float):
    """The DFlash2 selector on the workload's draft block (B requests, q_len
    positions, top 16 of the vocabulary, rank 256, hidden 5,120), random
    weights; greedy and MAP walks, CUDA events per call."""
    import speculative_decoding_target_gb300 as sv
    B, P, V = w.batch, w.q_len, w.vocab
    if P < 2:
        return None
    g = torch.Generator(device=dev).manual_seed(w.seed + 41)
    R, D = SELECT_RANK, SELECT_HIDDEN
    logits = torch.randn((B, P - 1, V), generator=g, device=dev) * 2
    boundary = torch.randint(0, V, (B,), generator=g, device=dev,
                             dtype=torch.int32)
    hidden = torch.randn((B, P - 1, D), generator=g, device=dev).to(
        torch.bfloat16)
    w_h = (torch.randn((R, D), generator=g, device=dev) / D ** 0.5).to(
        torch.bfloat16)
    code_a = (torch.randn((V, R), generator=g, device=dev) * 0.3).to(
        torch.bfloat16)
    code_b = (torch.randn((V, R), generator=g, device=dev) * 0.3).to(
        torch.bfloat16)
    out = torch.empty((B, P), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for mode in ("greedy", "map"):
        desc = sv._native.select_desc(logits, code_a, hidden,
                                      top=SELECT_TOP, mode=mode)
        ws = sv.alloc_workspace(sv._native.select_workspace_size(desc), dev)

        def call():
            sv.dflash2_select_into(desc, logits, boundary, hidden, w_h,
                                   code_a, code_b, out, None, None, None, ws,
                                   stream)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        res[mode + "_ms"] = round(statistics.mean(a.elapsed_time(b)
                                                  for a, b in evs), 5)
    nbytes = select_bytes(w)
    res.update({
        "shape": f"{B} requests x {P} positions, top {SELECT_TOP} of {V}, "
                 f"rank {R}, hidden {D}",
        "algorithmic_bytes": nbytes,
        "achieved_gbs_greedy": round(nbytes / (res["greedy_ms"] * 1e-3) / 1e9,
                                     1),
        "frac_of_peak_greedy": round(
            nbytes / (res["greedy_ms"] * 1e-3) / 1e9 / peak, 4),
        "gpu_launches": 3 * 2 * steps,
        "note": "three launches per call (after a counter reset): chunked "
                "top-K over the candidate logits (the streaming pass), the "
                "rank projection, the transition tables with the walk in "
                "each request's last table CTA",
    })
    return res


# ----------------------------------------------------------- CPU baseline --

def _oracle_step_estimate(w, host_inp, n_rows: int, n_acc_rows: int, rng):
    """Time the oracle on n_rows attention rows and n_acc_rows accept rows;
    return the extrapolated seconds of one full step."""
    import oracle
    bits = wl.to_numpy_bits
    total_rows = w.batch * w.q_len * w.num_q_heads
    rows = np.sort(rng.choice(total_rows, size=min(n_rows, total_rows),
                              replace=False)).astype(np.int64)
    fp8 = host_inp["k_scales"] is not None
    args = (bits(host_inp["q"]), bits(host_inp["k_pages"]),
            bits(host_inp["v_pages"]), host_inp["page_table"].numpy(),
            host_inp["seq_lens"].numpy())
    t = time.perf_counter()
    oracle.verify_attention(
        *args, num_kv_heads=w.num_kv_heads, scale=host_inp["scale"],
        k_scales=bits(host_inp["k_scales"]) if fp8 else None,
        v_scales=bits(host_inp["v_scales"]) if fp8 else None, rows=rows)
    t_attn = time.perf_counter() - t
    acc_total = w.batch * w.q_len
    nb = max(1, min(w.batch, n_acc_rows // w.q_len))
    lg = host_inp["logits"].numpy()[:nb * w.q_len]
    dr = host_inp["draft_ids"].numpy()[:nb]
    t = time.perf_counter()
    oracle.greedy_accept(lg, dr)
    t_acc = time.perf_counter() - t
    return (t_attn * total_rows / rows.size
            + t_acc * acc_total / (nb * w.q_len)), rows.size, nb * w.q_len


def cpu_baseline(w, host_inp, budget_s: float):
    import oracle
    rng = np.random.default_rng(w.seed)
    n = 8
    t0 = time.perf_counter()
    while True:
        est, nr, na = _oracle_step_estimate(w, host_inp, n, 2 * w.q_len, rng)
        spent = time.perf_counter() - t0
        total = w.batch * w.q_len * w.num_q_heads
        if spent > budget_s / 3 or nr >= total:
            break
        n = min(total, n * 4)
    return {"value": round(1.0 / est, 6), "unit": UNIT,
            "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"{nr} of {w.batch * w.q_len * w.num_q_heads} attention "
                      f"rows and {na} of {w.batch * w.q_len} logits rows of "
                      f"one step, extrapolated by row count "
                      f"({spent:.1f} s of CPU time)"}


# ------------------------------------------------------- reference arm --

def run_reference(args, w):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None, rank
    import oracle
    host_inp = wl.workload_inputs(w, device="cpu")
    rng = np.random.default_rng(w.seed + 1)
    n_rows = max(1, args.ref_rows)
    for _ in range(args.warmup):
        _oracle_step_estimate(w, host_inp, n_rows, w.q_len, rng)
    ests = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        est, nr, na = _oracle_step_estimate(w, host_inp, n_rows, w.q_len, rng)
        ests.append(est)
    spent = time.perf_counter() - t0
    value = 1.0 / statistics.mean(ests)
    sample = (f"{nr} of {w.batch * w.q_len * w.num_q_heads} attention rows "
              f"and {na} logits rows per step, extrapolated by row count")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 / value, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded, generated on the host)",
        "config": {"workload": w.name, "batch": w.batch, "q_len": w.q_len,
                   "prefix": w.prefix or "U[1024,131072]",
                   "page_size": w.page_size, "kv_dtype": w.kv_dtype},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT,
                         "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(spent, 2),
    }, rank


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(wl.ALL_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay each C-ABI call from a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-append", action="store_true",
                    help="skip the block KV append timing")
    ap.add_argument("--no-ragged", action="store_true",
                    help="skip the per-request width (ragged) step timing")
    ap.add_argument("--no-stochastic", action="store_true",
                    help="skip the rejection-sampling accept timing")
    ap.add_argument("--no-select", action="store_true",
                    help="skip the DFlash2 candidate selector timing")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--ref-rows", type=int, default=48)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = wl.ALL_WORKLOADS[args.workload]
    if args.impl == "reference":
        res, rank = run_reference(args, w)
    else:
        res, rank = run_gpu(args, w)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
