"""Seeded synthetic inputs for the target-verify step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no attention, no softmax, no acceptance rule).  Both the
CUDA library's tests/benchmark and the CPU oracle take their inputs from
here, so the two sides never exchange values computed by each other.

Shapes follow the target model the pages describe ("Qwen3.8-27B-FP8" page,
"Model specification": 24 query heads, 4 KV heads, head dimension 256,
vocabulary 248,320) and the paged KV pool of the serving stacks they discuss
("DFlash to dLLM self-spec, part 1", glossary entries req_to_token and
token_to_kv_pool).  The pool layout is [num_pages, Hkv, page_size, D]
(head-major inside a page); a request's pages are a random permutation of
the pool, pool slots that no request owns are filled with NaN so that any
out-of-range read poisons the result.

FP8 KV ("Qwen3.8-27B-FP8" page, "Implemented execution path": E4M3 cache
with per-token / per-KV-head FP16 scales over 64-channel blocks) is produced
by a fixed quantisation rule of this generator: for every (token, head,
64-channel block) scale = fp16(amax / 448) (1 when amax is 0), byte =
E4M3(x / scale) with round-to-nearest-even and saturation at +-448, using
torch's float8_e4m3fn conversion.  Parity never depends on this rule: both
sides consume the stored bytes and scales.

Logits are N(0, 4) fp32.  Drafts are planted: for each compared position j
independently, with probability p the draft is the row's argmax (torch
argmax, first index on ties), otherwise a uniform token other than it.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional, Sequence

import numpy as np
import torch

VOCAB = 248_320
NUM_Q_HEADS = 24
NUM_KV_HEADS = 4
HEAD_DIM = 256
BASE_SEED = 20261202

BF16_NAN_BITS = 0x7FC0
FP16_NAN_BITS = 0x7E00
E4M3_NAN_BYTE = 0x7F
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class VerifyWorkload:
    """One synthetic verify workload (attention + greedy accept)."""
    name: str
    batch: int
    q_len: int
    prefix: Optional[int]          # fixed prefix length, or None for a range
    prefix_range: Optional[tuple]  # (lo, hi) inclusive, uniform integers
    page_size: int
    kv_dtype: str                  # "bf16" or "fp8_e4m3"
    accept_p: float
    index: int
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM
    vocab: int = VOCAB

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index


# The five workloads: sizes, page sizes, dtypes and acceptance rates as the
# verify configurations of this project specify them.
WORKLOADS = {
    "b1_q8_p4k_ps16": VerifyWorkload("b1_q8_p4k_ps16", 1, 8, 4096, None, 16,
                                     "bf16", 0.5, 1),
    "b8_q8_p32k": VerifyWorkload("b8_q8_p32k", 8, 8, 32768, None, 64, "bf16",
                                 0.6, 2),
    "b1_q16_p256k": VerifyWorkload("b1_q16_p256k", 1, 16, 262144, None, 64,
                                   "bf16", 0.5, 3),
    "b32_q8_p1k128k_fp8": VerifyWorkload("b32_q8_p1k128k_fp8", 32, 8, None,
                                         (1024, 131072), 64, "fp8_e4m3", 0.5,
                                         4),
    "b4_q8_p512k": VerifyWorkload("b4_q8_p512k", 4, 8, 524288, None, 64,
                                  "bf16", 0.5, 5),
}
WORKLOAD_ORDER = list(WORKLOADS)

# Smaller cases of the same kernels for profiler captures that replay a
# launch many times: inputs still larger than L2, a few hundred MB on the
# device.  Not bench lines.
PROFILE_WORKLOADS = {
    "b8_q8_p16k_fp8": VerifyWorkload("b8_q8_p16k_fp8", 8, 8, 16384, None, 64,
                                     "fp8_e4m3", 0.5, 6),
}
ALL_WORKLOADS = {**WORKLOADS, **PROFILE_WORKLOADS}


def prefix_lengths(w: VerifyWorkload) -> List[int]:
    if w.prefix is not None:
        return [w.prefix] * w.batch
    g = torch.Generator().manual_seed(w.seed * 7 + 1)
    lo, hi = w.prefix_range
    return torch.randint(lo, hi + 1, (w.batch,), generator=g).tolist()


def kv_bytes(seq_lens: Sequence[int], num_kv_heads: int, head_dim: int,
             kv_dtype: str, include_scales: bool = True) -> int:
    """Algorithmic KV bytes one verify pass reads: every cached token of every
    request, K and V, every KV head (plus fp16 scales for FP8)."""
    tokens = int(sum(int(x) for x in seq_lens))
    if kv_dtype == "bf16":
        per = head_dim * 2
    else:
        per = head_dim + (2 * (head_dim // 64) if include_scales else 0)
    return tokens * num_kv_heads * 2 * per


def verify_flops(seq_lens: Sequence[int], q_len: int, num_q_heads: int,
                 head_dim: int) -> int:
    """QK^T plus PV multiply-adds (2 flops each) over the full cached
    length for every block row and query head."""
    tokens = int(sum(int(x) for x in seq_lens))
    return tokens * q_len * num_q_heads * head_dim * 4


def _bits16(x: torch.Tensor) -> torch.Tensor:
    return x.view(torch.int16)


def make_attention_inputs(*, batch: int, q_len: int, num_q_heads: int,
                          num_kv_heads: int, head_dim: int, page_size: int,
                          prefix_lens: Sequence[int], kv_dtype: str = "bf16",
                          seed: int = 0, device="cpu", spare_pages: int = -1,
                          shuffle: bool = True, poison: bool = True,
                          max_pages: Optional[int] = None,
                          value_std: float = 1.0,
                          fast_host: bool = False) -> dict:
    """Random verify-attention inputs in a paged pool.

    Returns a dict of tensors on ``device``:
      q [B, q_len, Hq, D] bf16; k_pages/v_pages [num_pages, Hkv, ps, D] bf16
      or uint8 (E4M3 bytes); k_scales/v_scales [num_pages, Hkv, ps, D/64]
      fp16 (FP8 only, else None); page_table int32 [B, max_pages] (-1 where
      unused); seq_lens int32 [B] = prefix + q_len; scale = 1/sqrt(D).

    fast_host: on the host, draw the K/V pools with numpy generators in
    threads (one stream per chunk of the pool) instead of torch's
    single-stream CPU generator, which takes minutes for pools of several
    GB.  The recipe (distribution, quantisation rule, layout, poisoning) is
    the same; the random values differ from a device-side draw.
    """
    device = torch.device(device)
    assert len(prefix_lens) == batch
    seq_lens = [int(p) + q_len for p in prefix_lens]
    pages_per = [math.ceil(s / page_size) for s in seq_lens]
    used = sum(pages_per)
    if spare_pages < 0:
        spare_pages = max(1, used // 16)
    num_pages = used + spare_pages
    if max_pages is None:
        max_pages = max(pages_per) if pages_per else 1
    assert max_pages >= max(pages_per, default=0)

    gcpu = torch.Generator().manual_seed(seed)
    perm = (torch.randperm(num_pages, generator=gcpu) if shuffle
            else torch.arange(num_pages))
    page_table = torch.full((batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        page_table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    spare = perm[off:]

    gdev = torch.Generator(device=device).manual_seed(seed + 1)
    q = (torch.randn((batch, q_len, num_q_heads, head_dim), generator=gdev,
                     device=device, dtype=torch.float32) * value_std
         ).to(torch.bfloat16)
    shape = (num_pages, num_kv_heads, page_size, head_dim)
    k_scales = v_scales = None
    host_fast = fast_host and device.type == "cpu"
    if kv_dtype == "bf16":
        k_pages = torch.empty(shape, dtype=torch.bfloat16, device=device)
        v_pages = torch.empty(shape, dtype=torch.bfloat16, device=device)
        for n, dst in enumerate((k_pages, v_pages)):
            if host_fast:
                _fill_randn_bf16_host(dst, seed * 4 + n, value_std)
            else:
                _fill_randn_bf16(dst, gdev, value_std)
    elif kv_dtype == "fp8_e4m3":
        assert head_dim % 64 == 0
        k_pages = torch.empty(shape, dtype=torch.uint8, device=device)
        v_pages = torch.empty(shape, dtype=torch.uint8, device=device)
        sshape = (num_pages, num_kv_heads, page_size, head_dim // 64)
        k_scales = torch.empty(sshape, dtype=torch.float16, device=device)
        v_scales = torch.empty(sshape, dtype=torch.float16, device=device)
        for n, (dst, sc) in enumerate(((k_pages, k_scales),
                                       (v_pages, v_scales))):
            if host_fast:
                _fill_randn_fp8_host(dst, sc, seed * 4 + n, value_std)
            else:
                _fill_randn_fp8(dst, sc, gdev, value_std)
    else:
        raise ValueError(kv_dtype)

    if poison:
        _poison(k_pages, v_pages, k_scales, v_scales, page_table, seq_lens,
                page_size, spare.to(device))
    return {
        "q": q, "k_pages": k_pages, "v_pages": v_pages,
        "k_scales": k_scales, "v_scales": v_scales,
        "page_table": page_table.to(device),
        "seq_lens": torch.tensor(seq_lens, dtype=torch.int32, device=device),
        "scale": 1.0 / math.sqrt(head_dim),
        "num_kv_heads": num_kv_heads, "kv_dtype": kv_dtype,
        "page_size": page_size,
    }


def _chunks(n: int, step: int):
    for s in range(0, n, step):
        yield s, min(n, s + step)


def _fill_randn_bf16(dst: torch.Tensor, g: torch.Generator, std: float):
    flat = dst.view(dst.shape[0], -1)
    step = max(1, (1 << 26) // max(1, flat.shape[1]))
    for s, e in _chunks(flat.shape[0], step):
        flat[s:e] = (torch.randn((e - s, flat.shape[1]), generator=g,
                                 device=dst.device) * std).to(torch.bfloat16)


def _fill_randn_fp8(dst: torch.Tensor, scales: torch.Tensor,
                    g: torch.Generator, std: float):
    npg = dst.shape[0]
    inner = dst.shape[1:]
    blocks = dst.shape[-1] // 64
    step = max(1, (1 << 25) // max(1, dst[0].numel()))
    for s, e in _chunks(npg, step):
        x = torch.randn((e - s,) + tuple(inner), generator=g,
                        device=dst.device) * std
        xb = x.view(e - s, inner[0], inner[1], blocks, 64)
        amax = xb.abs().amax(dim=-1)
        sc = torch.where(amax > 0, amax / E4M3_MAX,
                         torch.ones_like(amax)).to(torch.float16)
        y = (xb / sc.float().unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX)
        dst[s:e] = y.to(torch.float8_e4m3fn).view(torch.uint8).view(
            (e - s,) + tuple(inner))
        scales[s:e] = sc


def _host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


_HOST_CHUNK = 1 << 22


def _host_chunks(n: int, seed: int):
    """Chunks of a flat pool of n elements, each with its own numpy stream."""
    nch = (n + _HOST_CHUNK - 1) // _HOST_CHUNK
    return nch, np.random.SeedSequence(seed).spawn(max(1, nch))


def _fill_randn_bf16_host(dst: torch.Tensor, seed: int, std: float):
    """N(0, std^2) into a host bf16 tensor: float32 normals from numpy,
    rounded to bf16 to nearest-even on their bit patterns (finite values)."""
    out = dst.view(-1).view(torch.int16).numpy().view(np.uint16)
    nch, seqs = _host_chunks(out.size, seed)

    def work(c):
        s, e = c * _HOST_CHUNK, min(out.size, (c + 1) * _HOST_CHUNK)
        x = np.random.default_rng(seqs[c]).standard_normal(e - s,
                                                           dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        u = x.view(np.uint32)
        u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        out[s:e] = u >> np.uint32(16)

    with ThreadPoolExecutor(_host_threads()) as ex:
        list(ex.map(work, range(nch)))


def _fill_randn_fp8_host(dst: torch.Tensor, scales: torch.Tensor, seed: int,
                         std: float):
    """The FP8 rule of _fill_randn_fp8 on the host, a chunk of pages per
    numpy stream; torch converts to E4M3 (one intra-op thread per worker)."""
    npg = dst.shape[0]
    inner = tuple(dst.shape[1:])
    per_page = dst[0].numel()
    step = max(1, _HOST_CHUNK // max(1, per_page))
    nch = (npg + step - 1) // step
    seqs = np.random.SeedSequence(seed).spawn(max(1, nch))
    blocks = inner[-1] // 64

    def work(c):
        s, e = c * step, min(npg, (c + 1) * step)
        x = torch.from_numpy(np.random.default_rng(seqs[c]).standard_normal(
            (e - s,) + inner, dtype=np.float32))
        if std != 1.0:
            x *= std
        xb = x.view(e - s, inner[0], inner[1], blocks, 64)
        amax = xb.abs().amax(dim=-1)
        sc = torch.where(amax > 0, amax / E4M3_MAX,
                         torch.ones_like(amax)).to(torch.float16)
        y = (xb / sc.float().unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX)
        dst[s:e] = y.to(torch.float8_e4m3fn).view(torch.uint8).view(
            (e - s,) + inner)
        scales[s:e] = sc

    prev = torch.get_num_threads()
    torch.set_num_threads(1)
    try:
        with ThreadPoolExecutor(_host_threads()) as ex:
            list(ex.map(work, range(nch)))
    finally:
        torch.set_num_threads(prev)


def _poison(k_pages, v_pages, k_scales, v_scales, page_table, seq_lens,
            page_size, spare):
    fp8 = k_scales is not None
    tensors = [(k_pages, False), (v_pages, False)]
    if fp8:
        tensors += [(k_scales, True), (v_scales, True)]

    def raw(t, is_scale):
        # E4M3 bytes stay uint8; bf16 / fp16 are poisoned through their bits
        if fp8 and not is_scale:
            return t, E4M3_NAN_BYTE
        return t.view(torch.int16), (FP16_NAN_BITS if fp8 else BF16_NAN_BITS)

    if spare.numel():
        idx = spare.long()
        for t, is_scale in tensors:
            r, val = raw(t, is_scale)
            r[idx] = val
    for b, n_tok in enumerate(seq_lens):
        if n_tok <= 0:
            continue
        last = (n_tok - 1) // page_size
        first_bad = n_tok - last * page_size
        if first_bad < page_size:
            p = int(page_table[b, last])
            for t, is_scale in tensors:
                r, val = raw(t, is_scale)
                r[p, :, first_bad:] = val


def make_accept_inputs(*, batch: int, q_len: int, vocab: int, accept_p: float,
                       seed: int = 0, device="cpu", logit_std: float = 2.0):
    """fp32 logits [batch*q_len, vocab] ~ N(0, logit_std^2) and planted
    drafts int32 [batch, q_len] (column 0 = boundary token)."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(seed + 2)
    logits = torch.randn((batch * q_len, vocab), generator=g, device=device,
                         dtype=torch.float32) * logit_std
    am = logits.argmax(dim=-1).view(batch, q_len).to(torch.int32)
    u = torch.rand((batch, q_len), generator=g, device=device)
    other = torch.randint(0, max(1, vocab - 1), (batch, q_len), generator=g,
                          device=device, dtype=torch.int32)
    prev = torch.zeros_like(am)
    prev[:, 1:] = am[:, :-1]
    other = other + (other >= prev).to(torch.int32)  # uniform, != argmax
    drafts = torch.where(u < accept_p, prev, other)
    drafts[:, 0] = torch.randint(0, vocab, (batch,), generator=g,
                                 device=device, dtype=torch.int32)
    return {"logits": logits, "draft_ids": drafts.contiguous()}


def workload_inputs(w: VerifyWorkload, device="cpu", with_accept: bool = True,
                    fast_host: bool = False):
    """Inputs for one named workload (fast_host: see make_attention_inputs)."""
    attn = make_attention_inputs(
        batch=w.batch, q_len=w.q_len, num_q_heads=w.num_q_heads,
        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        page_size=w.page_size, prefix_lens=prefix_lengths(w),
        kv_dtype=w.kv_dtype, seed=w.seed, device=device, fast_host=fast_host)
    if with_accept:
        attn.update(make_accept_inputs(batch=w.batch, q_len=w.q_len,
                                       vocab=w.vocab, accept_p=w.accept_p,
                                       seed=w.seed, device=device))
    return attn


def to_numpy_bits(t: torch.Tensor):
    """Raw bits of a tensor as numpy (bf16/fp16 -> uint16, u8 stays)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
