#!/usr/bin/env python3
"""Benchmark of the target-verify step: paged GQA verify attention followed
by greedy acceptance, on seeded synthetic inputs, through the C ABI.

One step = spec_verify_attention over every request's verify block, then
spec_greedy_accept over the block's logits.

Headline workload (the largest, long-context configuration): batch 4, q_len
8, 24/4 heads, head_dim 256, 524,288-token prefixes in 64-token pages of a
permuted pool, bf16 KV (8.59 GB read per step); logits [32 x 248,320] fp32
with drafts planted at p = 0.5.  The same run times the four other verify
configurations (the "configs" key), each with its own roofline block: the
batch-1 4K-token and 256K-token cases both with a 512 MB L2 flush before
every step ("cold") and back to back ("warm"), the others (inputs larger
than L2) back to back.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica of the headline workload on its own GPU (the step has no cross-GPU
exchange), timing is the max over ranks, and value counts the steps of all
ranks; only rank 0 times the other configurations.

--impl reference times the CPU float64 oracle on the host cores instead
(rank 0 only): the K timed steps each compute a different 1/K of the
headline workload's attention rows and accept requests, so that together
they compute one whole verify step; value is whole steps per second.
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
DEFAULT_WORKLOAD = "b4_q8_p512k"
# our kernels per verify step: the split-KV attention kernel, the LSE merge
# kernel, the argmax/accept kernel (its last CTA per request finalises)
KERNEL_LAUNCHES_PER_STEP = 3
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20           # GB300 L2 (upper bound used for labels)
# configurations timed cold (L2 flushed before each step) and warm
COLD_AND_WARM = ("b1_q8_p4k_ps16", "b1_q16_p256k")

# DRAM traffic of the dominant kernel (the split-KV attention kernel):
# dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture, per
# algorithmic KV byte, keyed by the kernel and valid only while that
# kernel's sources still hash to the recorded value.  A workload other than
# the captured one gets the capture's bytes scaled by its algorithmic bytes
# (the traffic follows them: every KV byte is read once, and the partials
# are a small fixed share).
NCU_TRAFFIC = {
    "tc": {"source_hash": "4940d50b31ed6ff9", "captured_on": "b1_q16_p256k",
           "read": 1074314496, "write": 3420672,
           "algorithmic": 262160 * 4 * 1024},
    "fp8t": {"source_hash": "a3b122c912ef3bfd",
             "captured_on": "b8_q8_p16k_fp8",
             "read": 279394816, "write": 4690176,
             "algorithmic": 8 * 16392 * 4 * 528},
}

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


def traffic_per_launch(w, kv_b: int):
    """ncu DRAM bytes of one split-kernel launch on workload w (None when
    the kernel changed since the capture)."""
    kind = split_kernel_of(w)
    rec = NCU_TRAFFIC.get(kind)
    if not rec or rec["source_hash"] != kernel_source_hash(kind):
        return None, None
    per = (rec["read"] + rec["write"]) / rec["algorithmic"]
    how = ("captured on this workload" if rec["captured_on"] == w.name else
           f"captured on {rec['captured_on']}, scaled by algorithmic bytes")
    return int(round(per * kv_b)), how


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


def algorithmic_bytes(w: wl.VerifyWorkload, seq_lens=None):
    if seq_lens is None:
        seq_lens = [p + w.q_len for p in wl.prefix_lengths(w)]
    kv = wl.kv_bytes(seq_lens, w.num_kv_heads, w.head_dim, w.kv_dtype)
    logits = w.batch * w.q_len * w.vocab * 4
    return kv, logits


def config_of(w: wl.VerifyWorkload, ws_n: int, graph: bool = False) -> dict:
    """The workload description both arms print (identical dicts)."""
    kv_b, logit_b = algorithmic_bytes(w)
    return {
        "workload": w.name, "batch": w.batch, "q_len": w.q_len,
        "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim, "prefix": w.prefix or "U[1024,131072]",
        "page_size": w.page_size, "kv_dtype": w.kv_dtype,
        "vocab": w.vocab, "accept_p": w.accept_p, "seed": w.seed,
        "kv_bytes_per_step": kv_b, "logits_bytes_per_step": logit_b,
        "l2": (f"inputs larger than L2 ({(kv_b + logit_b) / 1e9:.3f} GB "
               "read per step), no flush" if kv_b + logit_b > L2_BYTES else
               f"inputs fit in L2 ({(kv_b + logit_b) / 1e9:.3f} GB read per "
               "step), steps back to back, no flush (warm)"),
        "parallelism": f"replicas x{ws_n}",
        "cuda_graph": bool(graph),
    }


def accept_statistics(accept_len, w: wl.VerifyWorkload) -> dict:
    """Mean accepted drafts and per-position survival of the synthetic
    logits.  Survival at position j is the share of requests that accepted
    at least j drafts; the survival rates sum to the mean accepted length
    ("Laguna S 2.1 DFlash accepting and FP8-KV result", acceptance and
    per-position survival).  Drafts are planted independently with
    probability p, so the expected accepted length is sum_j p^j."""
    a = [int(x) for x in accept_len]
    k = w.q_len - 1
    n = max(1, len(a))
    survival = [sum(1 for x in a if x >= j) / n for j in range(1, k + 1)]
    mean = sum(a) / n
    return {
        "requests": len(a), "mean_accept": round(mean, 6),
        "survival": [round(x, 6) for x in survival],
        "survival_sum": round(sum(survival), 6),
        "survival_sum_equals_mean": abs(sum(survival) - mean) < 1e-9,
        "expected_mean_accept": round(sum(w.accept_p ** j
                                          for j in range(1, k + 1)), 6),
        "commit_tokens_mean": round(mean + 1, 6),
    }


def tensor_digest(t) -> str:
    """sha256 of a tensor's bytes (small tensors), or of the int64 sums of
    its 32-bit words in 64 MiB chunks, computed where the tensor lives."""
    if t is None:
        return None
    b = t.detach().contiguous().view(-1).view(torch.uint8)
    h = hashlib.sha256()
    if b.numel() <= (64 << 20):
        h.update(b.cpu().numpy().tobytes())
        return h.hexdigest()[:16]
    words = b[: b.numel() // 4 * 4].view(torch.int32)
    chunk = 1 << 24
    full = words.numel() // chunk * chunk
    sums = words[:full].view(-1, chunk).sum(dim=1, dtype=torch.int64)
    h.update(sums.cpu().numpy().tobytes())
    h.update(words[full:].cpu().numpy().tobytes())
    h.update(b[words.numel() * 4:].cpu().numpy().tobytes())
    return "sum:" + h.hexdigest()[:16]


def input_digests(inp) -> dict:
    keys = ("q", "k_pages", "v_pages", "k_scales", "v_scales", "page_table",
            "seq_lens", "logits", "draft_ids")
    return {k: tensor_digest(inp.get(k)) for k in keys if inp.get(k) is not None}


# ----------------------------------------------------------------- GPU arm --

class VerifyStep:
    """Buffers and the step function of one workload on one device."""

    def __init__(self, w: wl.VerifyWorkload, inp: dict, dev):
        import speculative_decoding_target_gb300 as sv
        self.w, self.inp, self.dev = w, inp, dev
        self.desc = sv.desc_for(inp["q"], inp["k_pages"], inp["page_table"])
        self.attn_ws = sv.alloc_workspace(sv.verify_workspace_size(self.desc),
                                          dev)
        rows = w.batch * w.q_len
        self.acc_ws = sv.alloc_workspace(
            sv.accept_workspace_size(rows, w.vocab), dev)
        self.out = torch.empty_like(inp["q"])
        i32 = dict(dtype=torch.int32, device=dev)
        self.acc = torch.empty(w.batch, **i32)
        self.nxt = torch.empty(w.batch, **i32)
        self.toks = torch.empty((w.batch, w.q_len), **i32)
        self.stream = torch.cuda.current_stream(dev)

    def attention(self, stream=None):
        from speculative_decoding_target_gb300 import _native
        i = self.inp
        _native.verify_attention_into(
            self.desc, i["q"], i["k_pages"], i["v_pages"], i["k_scales"],
            i["v_scales"], i["page_table"], i["seq_lens"], i["scale"],
            self.out, self.attn_ws, stream or self.stream)

    def accept(self, stream=None):
        from speculative_decoding_target_gb300 import _native
        _native.greedy_accept_into(self.inp["logits"], self.inp["draft_ids"],
                                   self.acc, self.nxt, self.toks, self.acc_ws,
                                   stream or self.stream)

    def step(self, ev=None):
        if ev is not None:
            ev[0].record(self.stream)
        self.attention()
        if ev is not None:
            ev[1].record(self.stream)
        self.accept()
        if ev is not None:
            ev[2].record(self.stream)

    def timed(self, steps: int, flush=None):
        """Per-step (attention ms, accept ms, step ms) lists and the total
        ms of the loop.  With `flush` (a device buffer larger than L2) the
        buffer is rewritten before every step, outside its events."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
               for _ in range(steps)]
        torch.cuda.synchronize(self.dev)
        for k in range(steps):
            if flush is not None:
                flush.fill_(k & 0xFF)
            self.step(evs[k])
        torch.cuda.synchronize(self.dev)
        attn = [e[0].elapsed_time(e[1]) for e in evs]
        acc = [e[1].elapsed_time(e[2]) for e in evs]
        step = [e[0].elapsed_time(e[2]) for e in evs]
        total = evs[0][0].elapsed_time(evs[-1][2])
        return attn, acc, step, total


def roofline_block(w, kv_b: int, attn_ms: float, peak: float,
                   peak_kind: str) -> dict:
    achieved = kv_b / (attn_ms * 1e-3) / 1e9
    traffic, how = traffic_per_launch(w, kv_b)
    blk = {
        "kernel": "verify attention (split-KV kernel + LSE merge, one C-ABI "
                  "call)",
        "split_kernel": split_kernel_of(w),
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
        "peak_kind": peak_kind, "unit": "GB/s",
        "frac": round(achieved / peak, 4), "traffic": traffic,
        "algorithmic_bytes_per_launch": kv_b,
        "avg_launch_ms": round(attn_ms, 5),
    }
    if how:
        blk["traffic_note"] = how
    return blk


def measure_config(w: wl.VerifyWorkload, dev, steps: int, warmup: int,
                   peak: float, peak_kind: str, flush) -> dict:
    """Time one more configuration in the same run (rank 0): attention,
    accept and the whole step, cold (L2 flushed before each step) and warm
    for the batch-1 cases, back to back for the others."""
    inp = wl.workload_inputs(w, device=dev)
    vs = VerifyStep(w, inp, dev)
    for _ in range(warmup):
        vs.step()
    kv_b, logit_b = algorithmic_bytes(w, inp["seq_lens"].tolist())
    modes = ("cold", "warm") if w.name in COLD_AND_WARM else ("large",)
    rec = {"workload": w.name, "batch": w.batch, "q_len": w.q_len,
           "prefix": w.prefix or "U[1024,131072]", "page_size": w.page_size,
           "kv_dtype": w.kv_dtype, "seed": w.seed,
           "kv_bytes_per_step": kv_b, "logits_bytes_per_step": logit_b}
    for mode in modes:
        attn, acc, step, total = vs.timed(
            steps, flush if mode == "cold" else None)
        a, c = statistics.mean(attn), statistics.mean(acc)
        st = statistics.mean(step) if mode == "cold" else total / steps
        rec[mode] = {
            "l2": {"cold": f"{L2_FLUSH_BYTES >> 20} MB written before every "
                           "step, outside its events",
                   "warm": "steps back to back, no flush (KV and logits "
                           "partly or wholly L2-resident)",
                   "large": "inputs larger than L2, steps back to back, no "
                            "flush"}[mode],
            "steps_per_s": round(1e3 / st, 3), "step_ms": round(st, 5),
            "attention_ms": round(a, 5), "accept_ms": round(c, 5),
            "kv_read_gbs": round(kv_b / (a * 1e-3) / 1e9, 1),
            "frac": round(kv_b / (a * 1e-3) / 1e9 / peak, 4),
            "logits_gbs": round(logit_b / (c * 1e-3) / 1e9, 1),
        }
    main_mode = modes[0]
    rec["roofline"] = roofline_block(w, kv_b, rec[main_mode]["attention_ms"],
                                     peak, peak_kind)
    rec["roofline"]["l2"] = main_mode
    rec["acceptance"] = accept_statistics(vs.acc.cpu().tolist(), w)
    rec["input_digest"] = input_digests(inp)
    rec["gpu_launches"] = KERNEL_LAUNCHES_PER_STEP * (steps * len(modes) +
                                                      warmup)
    return rec, inp


def run_gpu(args, w: wl.VerifyWorkload):
    import speculative_decoding_target_gb300 as sv

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sv.load()

    inp = wl.workload_inputs(w, device=dev)
    seq_lens = inp["seq_lens"].tolist()
    vs = VerifyStep(w, inp, dev)
    stream = vs.stream

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    step = vs.step
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if args.graph:
        # one CUDA graph per C-ABI call, replayed in the timed loop: the
        # same kernels without the per-call host overhead
        g_attn, g_acc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g_attn, stream=side):
                vs.attention(side)
            with torch.cuda.graph(g_acc, stream=side):
                vs.accept(side)
        torch.cuda.synchronize(dev)

        def step(ev=None):
            if ev is not None:
                ev[0].record(stream)
            g_attn.replay()
            if ev is not None:
                ev[1].record(stream)
            g_acc.replay()
            if ev is not None:
                ev[2].record(stream)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    attn_ms = [e[0].elapsed_time(e[1]) for e in evs]
    acc_ms = [e[1].elapsed_time(e[2]) for e in evs]
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # end to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory and reads its results back
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, w, inp, vs.desc, vs.attn_ws, vs.acc_ws,
                          vs.out, stream, dev, ws_n, barrier)

    kv_b, logit_b = algorithmic_bytes(w, seq_lens)
    attn_avg_ms = statistics.mean(attn_ms)
    acc_avg_ms = statistics.mean(acc_ms)
    peak, peak_kind = measured_peaks()
    roof = roofline_block(w, kv_b, attn_avg_ms, peak, peak_kind)
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
        "config": config_of(w, ws_n, args.graph),
        "kv_read_gbs": roof["achieved"],
        "accept_ms": round(acc_avg_ms, 5),
        "logits_gbs": round(logit_b / (acc_avg_ms * 1e-3) / 1e9, 1),
        "roofline": roof,
        "gpu_launches": KERNEL_LAUNCHES_PER_STEP * args.steps,
        "kernel_source_hash": kernel_source_hash(split_kernel_of(w)),
        "clocks": clk,
    }
    if e2e is not None:
        result["e2e"] = e2e
    result["acceptance"] = accept_statistics(vs.acc.cpu().tolist(), w)
    result["input_digest"] = input_digests(inp)
    host_inp = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        host_inp = {k: (v.cpu() if torch.is_tensor(v) else v)
                    for k, v in inp.items()}
    if not args.main_only and rank == 0:
        del vs
        inp = None
        torch.cuda.empty_cache()
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        configs = {}
        extras_w = wl.WORKLOADS[args.extras_workload]
        extras_inp = None
        only = None if args.configs == "all" else {
            c for c in args.configs.split(",") if c and c != "none"}
        for name in wl.WORKLOAD_ORDER:
            if name == w.name or (only is not None and name not in only):
                continue
            cw = wl.WORKLOADS[name]
            rec, cinp = measure_config(cw, dev, args.steps, args.warmup,
                                       peak, peak_kind, flush)
            configs[name] = rec
            if name == extras_w.name:
                extras_inp = cinp
            del cinp
            torch.cuda.empty_cache()
        result["configs"] = configs
        if extras_inp is None and extras_w.name == w.name:
            extras_inp = wl.workload_inputs(w, device=dev)
        ex = {"workload": extras_w.name}
        if not args.no_append:
            ex["kv_append"] = measure_kv_append(extras_w, dev, args.steps,
                                                args.warmup)
        if not args.no_ragged:
            full = configs.get(extras_w.name, {}).get("large", {}).get(
                "attention_ms")
            ex["ragged"] = measure_ragged(extras_w, extras_inp, dev,
                                          args.steps, args.warmup, full)
        if not args.no_stochastic:
            ex["stochastic"] = measure_stochastic(extras_w, extras_inp, dev,
                                                  args.steps, args.warmup,
                                                  peak, flush)
        if not args.no_select:
            ex["dflash2_select"] = measure_select(extras_w, dev, args.steps,
                                                  args.warmup, peak, flush)
        result["next_rows"] = ex
        del extras_inp
        torch.cuda.empty_cache()
    if host_inp is not None:
        result["cpu_baseline"] = cpu_baseline(w, host_inp, args.cpu_seconds)
    if ws_n > 1:
        import torch.distributed as dist
        dist.barrier()
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
                   full_attn_ms=None):
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
        "attention_full_width_ms": (None if full_attn_ms is None
                                    else round(full_attn_ms, 5)),
        "accept_commit_ms": round(part[1], 5),
        "logits_bytes_read": rows * w.vocab * 4,
        "prepare_ms": round(part[2], 5),
        "gpu_launches": 4 * steps,
        "note": "attention streams the same KV whatever the widths (rows "
                "are free in the 128-row MMA tile); accept reads only the "
                "q_b logits rows of each request",
    }


# ------------------------------------------------------ stochastic verify --

def time_cold_calls(call, dev, steps: int, warmup: int, flush):
    """Device time of one call, cold: the call captured in a CUDA graph
    (eager calls would time the host's submission rate, since each call is
    shorter than its Python and ctypes overhead), replayed `steps` times
    with the L2 flushed before each replay, outside the replay's events.
    Returns (mean, median) in ms."""
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        call(stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call(side)
    torch.cuda.synchronize(dev)
    for _ in range(warmup):
        graph.replay()
    evs = [(torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for k, (a, b) in enumerate(evs):
        flush.fill_(k & 0xFF)
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in evs]
    return statistics.mean(ms), statistics.median(ms)


def measure_stochastic(w: wl.VerifyWorkload, inp, dev, steps: int,
                       warmup: int, peak: float, flush):
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
    out = {}
    for name, dp in (("greedy_drafts", None), ("draft_probs", probs)):
        def call(st, dp=dp):
            sv.stochastic_accept_into(inp["logits"], inp["draft_ids"], dp,
                                      None, temp, ua, us, None, None, acc,
                                      nxt, toks, ws, st)
        mean, med = time_cold_calls(call, dev, steps, warmup, flush)
        out[name + "_ms"] = round(mean, 5)
        out[name + "_median_ms"] = round(med, 5)
    logit_bytes = B * q * V * 4
    out.update({
        "logits_bytes": logit_bytes,
        "logits_gbs_greedy_drafts": round(
            logit_bytes / (out["greedy_drafts_ms"] * 1e-3) / 1e9, 1),
        "frac_of_peak_greedy_drafts": round(
            logit_bytes / (out["greedy_drafts_ms"] * 1e-3) / 1e9 / peak, 4),
        "gpu_launches": (2 + 3) * steps,
        "timing": "per call: CUDA graph replay, L2 flushed (512 MB written) "
                  "before each call outside its events",
        "note": "one streaming pass over the logits (softmax statistics), "
                "then the draw; with full draft distributions a pass over "
                "the rejection row's chunks (residual weights) in between "
                "(a greedy drafter's residual follows from the statistics); "
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
                   peak: float, flush):
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
    res = {}
    for mode in ("greedy", "map"):
        desc = sv._native.select_desc(logits, code_a, hidden,
                                      top=SELECT_TOP, mode=mode)
        ws = sv.alloc_workspace(sv._native.select_workspace_size(desc), dev)

        def call(st, desc=desc, ws=ws):
            sv.dflash2_select_into(desc, logits, boundary, hidden, w_h,
                                   code_a, code_b, out, None, None, None, ws,
                                   st)
        mean, med = time_cold_calls(call, dev, steps, warmup, flush)
        res[mode + "_ms"] = round(mean, 5)
        res[mode + "_median_ms"] = round(med, 5)
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
        "timing": "per call: CUDA graph replay, L2 flushed (512 MB written) "
                  "before each call outside its events",
        "note": "three launches per call (after a counter reset): chunked "
                "top-K over the candidate logits (the streaming pass), the "
                "rank projection, the transition tables with the walk in "
                "each request's last table CTA",
    })
    return res


# ----------------------------------------------------------- CPU baseline --

def _oracle_rows(w, host_inp, rows):
    """The oracle's attention over the given flat rows (b*q_len + i)*Hq + h."""
    import oracle
    bits = wl.to_numpy_bits
    fp8 = host_inp["k_scales"] is not None
    return oracle.verify_attention(
        bits(host_inp["q"]), bits(host_inp["k_pages"]),
        bits(host_inp["v_pages"]), host_inp["page_table"].numpy(),
        host_inp["seq_lens"].numpy(), num_kv_heads=w.num_kv_heads,
        scale=host_inp["scale"],
        k_scales=bits(host_inp["k_scales"]) if fp8 else None,
        v_scales=bits(host_inp["v_scales"]) if fp8 else None,
        rows=np.asarray(rows, np.int64))


def _oracle_accept(w, host_inp, requests):
    import oracle
    if len(requests) == 0:
        return
    lo, hi = int(requests[0]), int(requests[-1]) + 1
    lg = host_inp["logits"].numpy()[lo * w.q_len:hi * w.q_len]
    oracle.greedy_accept(lg, host_inp["draft_ids"].numpy()[lo:hi])


def cpu_baseline(w, host_inp, budget_s: float):
    """The oracle as it stands on a bounded sample of one step: a growing
    random sample of attention rows (and the accept of a proportional share
    of the requests) until about budget_s seconds are spent, extrapolated to
    the whole step by row count."""
    import oracle
    rng = np.random.default_rng(w.seed)
    total = w.batch * w.q_len * w.num_q_heads
    perm = rng.permutation(total)
    n, spent, t_rows, n_done = 8, 0.0, 0.0, 0
    while True:
        rows = np.sort(perm[n_done:n_done + n])
        t = time.perf_counter()
        _oracle_rows(w, host_inp, rows)
        dt = time.perf_counter() - t
        t_rows += dt
        n_done += rows.size
        spent += dt
        per_row = t_rows / n_done
        left = total - n_done
        if left == 0 or spent + per_row * min(left, 4 * n) > budget_s:
            break
        n = min(left, 4 * n)
    nreq = max(1, round(w.batch * n_done / total))
    t = time.perf_counter()
    _oracle_accept(w, host_inp, np.arange(nreq))
    t_acc = time.perf_counter() - t
    est = per_row * total + t_acc * w.batch / nreq
    return {"value": round(1.0 / est, 6), "unit": UNIT,
            "cores": oracle.default_threads(), "kind": "oracle",
            "sample": f"{n_done} of {total} attention rows (random) and the "
                      f"accept of {nreq} of {w.batch} requests of one step, "
                      f"extrapolated by row count ({spent + t_acc:.1f} s of "
                      f"oracle time)"}


# ------------------------------------------------------- reference arm --

def run_reference(args, w):
    """The CPU float64 oracle as the reference arm.  The K timed steps each
    compute a different 1/K of the workload's attention rows and accept
    requests (contiguous slices), so together they compute one whole verify
    step: ms_per_step is the time of one slice, value is whole verify steps
    per second (1 / the sum of the K slice times).  Warm-up steps compute a
    few rows each.  Inputs are drawn on the host with the workload's recipe
    and seed (the random values differ from the device-side draw)."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None, rank
    import oracle
    t_gen = time.perf_counter()
    host_inp = wl.workload_inputs(w, device="cpu", fast_host=True)
    t_gen = time.perf_counter() - t_gen
    total = w.batch * w.q_len * w.num_q_heads
    K = max(1, args.steps)
    row_slices = np.array_split(np.arange(total, dtype=np.int64), K)
    req_slices = np.array_split(np.arange(w.batch, dtype=np.int64), K)
    for k in range(args.warmup):
        _oracle_rows(w, host_inp, row_slices[k % K][:8])
    times = []
    for k in range(K):
        t = time.perf_counter()
        if row_slices[k].size:
            _oracle_rows(w, host_inp, row_slices[k])
        _oracle_accept(w, host_inp, req_slices[k])
        times.append(time.perf_counter() - t)
    whole = sum(times)
    value = 1.0 / whole
    sample = (f"each of the {K} timed steps computes 1/{K} of the "
              f"{total} attention rows and of the {w.batch} accept requests; "
              f"the {K} together compute one whole verify step in "
              f"{whole:.2f} s")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * whole / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded, generated on the host)",
        "config": config_of(w, ws_n, args.graph),
        "step_fraction": round(1.0 / K, 6),
        "value_basis": "whole verify steps per second: 1 / (sum of the K "
                       "slice times)",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT,
                         "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "input_generation_s": round(t_gen, 2),
        "timed_s": round(whole, 2),
    }, rank


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(wl.ALL_WORKLOADS))
    ap.add_argument("--main-only", action="store_true",
                    help="time only --workload (no other configurations, "
                         "no next-row timings)")
    ap.add_argument("--extras-workload", default="b8_q8_p32k",
                    choices=list(wl.WORKLOADS),
                    help="workload whose shapes the next-row timings use")
    ap.add_argument("--configs", default="all",
                    help="comma list of the other configurations to time "
                         "after the headline ('all', or 'none' for the "
                         "widened rows alone)")
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
