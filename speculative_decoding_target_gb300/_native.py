"""ctypes binding of libspecverify.so (argument marshalling only).

Every step of the verify path runs in the library's CUDA kernels; this module
only turns torch tensors into device pointers and sizes, and the current torch
stream into a cudaStream_t.  There is no fallback: if the library is missing
or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_ARG = -1
SPEC_ERR_ALIGN = -2
SPEC_ERR_WORKSPACE = -3
SPEC_ERR_UNSUPPORTED = -4
SPEC_ERR_CUDA = -5
SPEC_KV_BF16 = 0
SPEC_KV_FP8_E4M3 = 1
SPEC_FLAG_CHECKED = 1
SPEC_STATUS_BAD_PAGE = 1
SPEC_STATUS_TIMEOUT = 2
SPEC_STATUS_NO_SLOT = 4
WIDTH_POLICIES = {"fixed": 0, "ewma": 1, "doubling": 2}

EXPORTED = (
    "spec_verify_workspace_size", "spec_verify_attention",
    "spec_verify_status", "spec_accept_workspace_size", "spec_greedy_accept",
    "spec_last_error", "spec_version", "spec_verify_attention_noalloc",
    "spec_kv_append", "spec_greedy_accept_commit", "spec_prepare_next_block",
    "spec_stochastic_workspace_size", "spec_stochastic_accept",
    "spec_select_workspace_size", "spec_dflash2_select",
    "spec_verify_set_wait_limit",
)
SELECT_MODES = {"greedy": 0, "map": 1}
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class SpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"spec_verify error {code}: {msg}")
        self.code = code


class AttnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("q_lens", ctypes.c_void_p)]


class SelectDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("positions", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("top", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("mode", ctypes.c_int32)]


class WidthPolicy(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("q_max", ctypes.c_int32),
                ("min_width", ctypes.c_int32), ("mask_id", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("offset", ctypes.c_float)]


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} not found: build it with "
            "`python -m speculative_decoding_target_gb300.build`")
    lib = ctypes.CDLL(path)
    P, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
    sz = ctypes.c_size_t
    lib.spec_verify_workspace_size.argtypes = [ctypes.POINTER(AttnDesc)]
    lib.spec_verify_workspace_size.restype = sz
    lib.spec_verify_attention.argtypes = [
        ctypes.POINTER(AttnDesc), P, P, P, P, P, P, P, ctypes.c_float, P, P,
        sz, P]
    lib.spec_verify_attention.restype = ctypes.c_int
    lib.spec_verify_attention_noalloc.argtypes = [
        ctypes.POINTER(AttnDesc), P, P, P, P, P, P, P, ctypes.c_float, P, P]
    lib.spec_verify_attention_noalloc.restype = ctypes.c_int
    lib.spec_kv_append.argtypes = [ctypes.POINTER(AttnDesc), P, P, P, P, P,
                                   P, P, P, P, P, P, P]
    lib.spec_kv_append.restype = ctypes.c_int
    lib.spec_verify_set_wait_limit.argtypes = [ctypes.c_int64]
    lib.spec_verify_set_wait_limit.restype = ctypes.c_int
    lib.spec_verify_status.argtypes = [P, ctypes.POINTER(u32), i32, P]
    lib.spec_verify_status.restype = ctypes.c_int
    lib.spec_accept_workspace_size.argtypes = [i32, i32]
    lib.spec_accept_workspace_size.restype = sz
    lib.spec_greedy_accept.argtypes = [P, P, i32, i32, i32, P, P, P, P, sz, P]
    lib.spec_greedy_accept.restype = ctypes.c_int
    lib.spec_greedy_accept_commit.argtypes = [P, P, P, i32, i32, i32, P, P, P,
                                              P, P, P, sz, P]
    lib.spec_greedy_accept_commit.restype = ctypes.c_int
    lib.spec_prepare_next_block.argtypes = [
        ctypes.POINTER(WidthPolicy), i32, P, P, P, P, P, P, i32, i32, i32, P,
        P, P, P, P, P, P]
    lib.spec_prepare_next_block.restype = ctypes.c_int
    lib.spec_stochastic_workspace_size.argtypes = [i32, i32, i32]
    lib.spec_stochastic_workspace_size.restype = sz
    lib.spec_stochastic_accept.argtypes = [P, P, P, P, i32, i32, i32, P, P, P,
                                           P, P, P, P, P, P, sz, P]
    lib.spec_stochastic_accept.restype = ctypes.c_int
    lib.spec_select_workspace_size.argtypes = [ctypes.POINTER(SelectDesc)]
    lib.spec_select_workspace_size.restype = sz
    lib.spec_dflash2_select.argtypes = [ctypes.POINTER(SelectDesc), P, P, P,
                                        P, P, P, P, P, P, P, P, sz, P]
    lib.spec_dflash2_select.restype = ctypes.c_int
    lib.spec_last_error.argtypes = []
    lib.spec_last_error.restype = ctypes.c_char_p
    lib.spec_version.argtypes = []
    lib.spec_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(rc: int):
    if rc != SPEC_OK:
        raise SpecError(rc, load().spec_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(*, batch, q_len, num_q_heads, num_kv_heads, head_dim,
              page_size, num_pages, max_pages_per_seq, kv_dtype="bf16",
              checked=False, q_lens: Optional[torch.Tensor] = None) -> AttnDesc:
    """q_lens: optional int32 device tensor [B] of per-request block rows."""
    return AttnDesc(batch, q_len, num_q_heads, num_kv_heads, head_dim,
                    page_size, num_pages, max_pages_per_seq,
                    SPEC_KV_BF16 if kv_dtype == "bf16" else SPEC_KV_FP8_E4M3,
                    SPEC_FLAG_CHECKED if checked else 0,
                    None if q_lens is None else q_lens.data_ptr())


def desc_for(q: torch.Tensor, k_pages: torch.Tensor,
             page_table: torch.Tensor, checked: bool = False,
             q_lens: Optional[torch.Tensor] = None) -> AttnDesc:
    B, q_len, hq, d = q.shape
    num_pages, hkv, ps, d2 = k_pages.shape
    assert d2 == d
    return make_desc(batch=B, q_len=q_len, num_q_heads=hq, num_kv_heads=hkv,
                     head_dim=d, page_size=ps, num_pages=num_pages,
                     max_pages_per_seq=page_table.shape[1],
                     kv_dtype="fp8" if k_pages.dtype == torch.uint8 else "bf16",
                     checked=checked, q_lens=q_lens)


def verify_workspace_size(desc: AttnDesc) -> int:
    n = load().spec_verify_workspace_size(ctypes.byref(desc))
    if n == 0:
        raise SpecError(SPEC_ERR_ARG, load().spec_last_error().decode())
    return int(n)


def accept_workspace_size(rows: int, vocab: int) -> int:
    return int(load().spec_accept_workspace_size(rows, vocab))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator hands out 512-byte aligned blocks
    return torch.empty(max(1, nbytes), dtype=torch.uint8, device=device)


def verify_attention_into(desc: AttnDesc, q, k_pages, v_pages, k_scales,
                          v_scales, page_table, seq_lens, scale: float, out,
                          workspace: torch.Tensor, stream=None) -> None:
    _check(load().spec_verify_attention(
        ctypes.byref(desc), _ptr(q), _ptr(k_pages), _ptr(v_pages),
        _ptr(k_scales), _ptr(v_scales), _ptr(page_table), _ptr(seq_lens),
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream)))


def verify_attention(q, k_pages, v_pages, page_table, seq_lens, *,
                     scale: float, k_scales=None, v_scales=None,
                     out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     checked: bool = False, q_lens=None,
                     stream=None) -> torch.Tensor:
    """Verify attention on device tensors; returns out bf16 [B, q_len, Hq, D]
    (q_lens: optional int32 [B] rows per request of a block padded to
    q_len)."""
    desc = desc_for(q, k_pages, page_table, checked, q_lens)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(verify_workspace_size(desc), q.device)
    verify_attention_into(desc, q, k_pages, v_pages, k_scales, v_scales,
                          page_table, seq_lens, scale, out, workspace, stream)
    return out


def verify_attention_noalloc(q, k_pages, v_pages, page_table, seq_lens, *,
                             scale: float, k_scales=None, v_scales=None,
                             out: Optional[torch.Tensor] = None,
                             q_lens=None, stream=None) -> torch.Tensor:
    """Verify attention with the library's fixed scratch instead of a
    workspace (for callers that cannot allocate device memory)."""
    desc = desc_for(q, k_pages, page_table, q_lens=q_lens)
    if out is None:
        out = torch.empty_like(q)
    _check(load().spec_verify_attention_noalloc(
        ctypes.byref(desc), _ptr(q), _ptr(k_pages), _ptr(v_pages),
        _ptr(k_scales), _ptr(v_scales), _ptr(page_table), _ptr(seq_lens),
        float(scale), _ptr(out), _stream(stream)))
    return out


def kv_append(k_new, v_new, k_pages, v_pages, page_table, seq_lens, *,
              k_scales=None, v_scales=None, positions=None, cache_loc=None,
              checked: bool = False, workspace=None, q_lens=None,
              stream=None):
    """Append the verify block's K/V (bf16 [B, q_len, Hkv, D]) to the paged
    pool in place (quantised on write for an FP8 pool); fills the optional
    positions (int32 [B, q_len]) and cache_loc (int64 [B, q_len])."""
    B, q_len, hkv, d = k_new.shape
    num_pages, hkv2, ps, _ = k_pages.shape
    desc = make_desc(batch=B, q_len=q_len, num_q_heads=hkv, num_kv_heads=hkv,
                     head_dim=d, page_size=ps, num_pages=num_pages,
                     max_pages_per_seq=page_table.shape[1],
                     kv_dtype="fp8" if k_pages.dtype == torch.uint8 else "bf16",
                     checked=checked, q_lens=q_lens)
    _check(load().spec_kv_append(
        ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
        _ptr(v_pages), _ptr(k_scales), _ptr(v_scales), _ptr(page_table),
        _ptr(seq_lens), _ptr(positions), _ptr(cache_loc), _ptr(workspace),
        _stream(stream)))


def set_wait_limit(cycles: int) -> None:
    """Main-loop wait bound (SM clock cycles) of the split kernels for calls
    with checked=True; 0 restores the default.  A test hook for the timeout
    path."""
    _check(load().spec_verify_set_wait_limit(int(cycles)))


def verify_status(workspace: torch.Tensor, clear: bool = True,
                  stream=None) -> int:
    st = ctypes.c_uint32(0)
    _check(load().spec_verify_status(_ptr(workspace), ctypes.byref(st),
                                     int(clear), _stream(stream)))
    return int(st.value)


def greedy_accept_into(logits, draft_ids, accept_len, next_token, out_tokens,
                       workspace: torch.Tensor, stream=None) -> None:
    B, q_len = draft_ids.shape
    _check(load().spec_greedy_accept(
        _ptr(logits), _ptr(draft_ids), B, q_len, logits.shape[-1],
        _ptr(accept_len), _ptr(next_token), _ptr(out_tokens),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def greedy_accept_commit_into(logits, draft_ids, q_lens, seq_lens,
                              new_seq_lens, accept_len, next_token, out_tokens,
                              workspace: torch.Tensor, stream=None) -> None:
    B, q_len = draft_ids.shape
    _check(load().spec_greedy_accept_commit(
        _ptr(logits), _ptr(draft_ids), _ptr(q_lens), B, q_len,
        logits.shape[-1], _ptr(seq_lens), _ptr(new_seq_lens),
        _ptr(accept_len), _ptr(next_token), _ptr(out_tokens),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def greedy_accept_commit(logits, draft_ids, q_lens, seq_lens, *,
                         workspace: Optional[torch.Tensor] = None,
                         stream=None):
    """Greedy accept with per-request widths and the committed cache length.
    Returns (accept_len, next_token, out_tokens, new_seq_lens)."""
    B, q_len = draft_ids.shape
    dev = logits.device
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty((B, q_len), dtype=torch.int32, device=dev)
    new = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(
            accept_workspace_size(B * q_len, logits.shape[-1]), dev)
    greedy_accept_commit_into(logits, draft_ids, q_lens, seq_lens, new, acc,
                              nxt, toks, workspace, stream)
    return acc, nxt, toks, new


def width_policy(policy: str, q_max: int, *, min_width: int = 2,
                 alpha: float = 0.5, offset: float = 1.5,
                 mask_id: int = 0) -> WidthPolicy:
    return WidthPolicy(WIDTH_POLICIES[policy], q_max, min_width, mask_id,
                       alpha, offset)


def prepare_next_block_into(pol: WidthPolicy, q_lens, accept_len, next_token,
                            new_seq_lens, state, page_table, page_size: int,
                            num_pages: int, next_q_lens, next_seq_lens,
                            block_ids=None, positions=None, cache_loc=None,
                            status=None, stream=None) -> None:
    B = accept_len.shape[0]
    _check(load().spec_prepare_next_block(
        ctypes.byref(pol), B, _ptr(q_lens), _ptr(accept_len),
        _ptr(next_token), _ptr(new_seq_lens), _ptr(state), _ptr(page_table),
        page_table.shape[1], page_size, num_pages, _ptr(next_q_lens),
        _ptr(next_seq_lens), _ptr(block_ids), _ptr(positions),
        _ptr(cache_loc), _ptr(status), _stream(stream)))


def prepare_next_block(pol: WidthPolicy, q_lens, accept_len, next_token,
                       new_seq_lens, state, page_table, *, page_size: int,
                       num_pages: int, status=None, stream=None):
    """Next widths and next-block layout on the device (state updated in
    place).  Returns dict of next_q_lens, next_seq_lens, block_ids,
    positions, cache_loc."""
    B = accept_len.shape[0]
    dev = accept_len.device
    out = {"next_q_lens": torch.empty(B, dtype=torch.int32, device=dev),
           "next_seq_lens": torch.empty(B, dtype=torch.int32, device=dev),
           "block_ids": torch.empty((B, pol.q_max), dtype=torch.int32,
                                    device=dev),
           "positions": torch.empty((B, pol.q_max), dtype=torch.int32,
                                    device=dev),
           "cache_loc": torch.empty((B, pol.q_max), dtype=torch.int64,
                                    device=dev)}
    prepare_next_block_into(pol, q_lens, accept_len, next_token, new_seq_lens,
                            state, page_table, page_size, num_pages,
                            out["next_q_lens"], out["next_seq_lens"],
                            out["block_ids"], out["positions"],
                            out["cache_loc"], status, stream)
    return out


def stochastic_workspace_size(batch: int, q_len: int, vocab: int) -> int:
    return int(load().spec_stochastic_workspace_size(batch, q_len, vocab))


def stochastic_accept_into(logits, draft_ids, draft_probs, q_lens,
                           temperature, u_accept, u_sample, seq_lens,
                           new_seq_lens, accept_len, next_token, out_tokens,
                           workspace: torch.Tensor, stream=None) -> None:
    B, q_len = draft_ids.shape
    _check(load().spec_stochastic_accept(
        _ptr(logits), _ptr(draft_ids), _ptr(draft_probs), _ptr(q_lens), B,
        q_len, logits.shape[-1], _ptr(temperature), _ptr(u_accept),
        _ptr(u_sample), _ptr(seq_lens), _ptr(new_seq_lens), _ptr(accept_len),
        _ptr(next_token), _ptr(out_tokens), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def stochastic_accept(logits, draft_ids, temperature, u_accept, u_sample, *,
                      draft_probs=None, q_lens=None, seq_lens=None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """Rejection-sampling verify.  Returns (accept_len, next_token,
    out_tokens, new_seq_lens or None)."""
    B, q_len = draft_ids.shape
    dev = logits.device
    i32 = dict(dtype=torch.int32, device=dev)
    acc, nxt = torch.empty(B, **i32), torch.empty(B, **i32)
    toks = torch.empty((B, q_len), **i32)
    new = torch.empty(B, **i32) if seq_lens is not None else None
    if workspace is None:
        workspace = alloc_workspace(
            stochastic_workspace_size(B, q_len, logits.shape[-1]), dev)
    stochastic_accept_into(logits, draft_ids, draft_probs, q_lens,
                           temperature, u_accept, u_sample, seq_lens, new,
                           acc, nxt, toks, workspace, stream)
    return acc, nxt, toks, new


def select_desc(cand_logits, code_a, hidden, *, top: int = 16,
                mode: str = "greedy") -> SelectDesc:
    B, P1, V = cand_logits.shape
    return SelectDesc(B, P1 + 1, V, top, code_a.shape[1], hidden.shape[2],
                      SELECT_MODES[mode])


def select_workspace_size(desc: SelectDesc) -> int:
    n = load().spec_select_workspace_size(ctypes.byref(desc))
    if n == 0:
        raise SpecError(SPEC_ERR_ARG, load().spec_last_error().decode())
    return int(n)


def dflash2_select_into(desc: SelectDesc, cand_logits, boundary, hidden, w_h,
                        code_a, code_b, draft_ids, cand_ids, cand_logit,
                        trans, workspace: torch.Tensor, stream=None) -> None:
    _check(load().spec_dflash2_select(
        ctypes.byref(desc), _ptr(cand_logits), _ptr(boundary), _ptr(hidden),
        _ptr(w_h), _ptr(code_a), _ptr(code_b), _ptr(draft_ids),
        _ptr(cand_ids), _ptr(cand_logit), _ptr(trans), _ptr(workspace),
        workspace.numel(), _stream(stream)))


def dflash2_select(cand_logits, boundary, hidden, w_h, code_a, code_b, *,
                   top: int = 16, mode: str = "greedy",
                   workspace: Optional[torch.Tensor] = None, stream=None):
    """DFlash2 candidate selection on device tensors.  Returns dict of
    draft_ids [B, P], cand_ids [B, P-1, K], cand_logit [B, P-1, K] and
    trans [B, P-1, K, K]."""
    desc = select_desc(cand_logits, code_a, hidden, top=top, mode=mode)
    B, P1 = cand_logits.shape[:2]
    dev = cand_logits.device
    out = {"draft_ids": torch.empty((B, P1 + 1), dtype=torch.int32,
                                    device=dev),
           "cand_ids": torch.empty((B, P1, top), dtype=torch.int32,
                                   device=dev),
           "cand_logit": torch.empty((B, P1, top), device=dev),
           "trans": torch.empty((B, P1, top, top), device=dev)}
    if workspace is None:
        workspace = alloc_workspace(select_workspace_size(desc), dev)
    dflash2_select_into(desc, cand_logits, boundary, hidden, w_h, code_a,
                        code_b, out["draft_ids"], out["cand_ids"],
                        out["cand_logit"], out["trans"], workspace, stream)
    return out


def greedy_accept(logits: torch.Tensor, draft_ids: torch.Tensor, *,
                  workspace: Optional[torch.Tensor] = None,
                  with_tokens: bool = True, stream=None):
    """Returns (accept_len [B], next_token [B], out_tokens [B, q_len] or None)."""
    B, q_len = draft_ids.shape
    dev = logits.device
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    toks = (torch.empty((B, q_len), dtype=torch.int32, device=dev)
            if with_tokens else None)
    if workspace is None:
        workspace = alloc_workspace(
            accept_workspace_size(B * q_len, logits.shape[-1]), dev)
    greedy_accept_into(logits, draft_ids, acc, nxt, toks, workspace, stream)
    return acc, nxt, toks
