"""CPU float64 oracle for the target-verify step (test infrastructure only).

This package is TEST INFRASTRUCTURE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product library (``speculative_decoding_target_gb300``) never imports,
links or calls anything here, and this package imports nothing from it: the
two share no code.  Inputs reach both sides from the seeded generators in
``speculative_decoding_target_gb300.workloads``, which hold none of the
method's arithmetic.

The arithmetic lives in ``spec_oracle.c`` (plain C, float64, OpenMP over
output rows only); this module compiles it with gcc and wraps it with
ctypes.  Every function cites the passage it follows in the C file.

Pins (see ``tests/test_oracle.py`` and ``tests/test_oracle_append.py``):
the E4M3 / fp16 encoders against torch's float8_e4m3fn and numpy's float16
conversions, torch float64 scaled-dot-product
attention on gathered dense K/V, torch's float8_e4m3fn and numpy's float16
decoders on every bit pattern, closed forms (identical keys, dominant key,
two-key sigmoid), the invariants the pages fix (q_len=1 equals decode, row i
equals a q_len=1 call over prefix + drafts 1..i, merge of split partials
equals the unsplit result, permuted pages and poisoned slots change nothing),
numpy argmax on exhaustive tiny tie patterns, the pages' worked accept
examples, and a serial-greedy simulation of the commit stream.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libspec_oracle.so")
_lib = None

ORACLE_OK = 0
ORACLE_ERR_ARG = -1
ORACLE_ERR_PAGE = -2
ORACLE_ERR_NOMEM = -3


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into a shared library with gcc (portable flags)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # no contraction into fused multiply-adds: the float32 steps the
    # oracle states (quantisation, the width EWMA) are rounded one by one
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_verify_attention.argtypes = [
        i32, i32, i32, i32, i32, i32, i32, i32, i32,
        P, P, P, P, P, P, P, P, f64, P, i64, i64, i64, P, P, i32]
    lib.oracle_verify_attention.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [i32, i32, P, P, P, P]
    lib.oracle_lse_merge.restype = None
    lib.oracle_greedy_accept.argtypes = [P, P, P, i32, i32, i64, P, P, P, P,
                                         P, P, i32]
    lib.oracle_greedy_accept.restype = ctypes.c_int
    for name in ("oracle_decode_bf16", "oracle_decode_fp16"):
        getattr(lib, name).argtypes = [P, i64, P]
        getattr(lib, name).restype = None
    lib.oracle_decode_e4m3.argtypes = [P, i64, P]
    lib.oracle_decode_e4m3.restype = None
    for name in ("oracle_encode_fp16", "oracle_encode_e4m3"):
        getattr(lib, name).argtypes = [P, i64, P]
        getattr(lib, name).restype = None
    lib.oracle_kv_append.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                     P, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_kv_append.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.oracle_prepare_next_block.argtypes = [
        i32, i32, i32, f32, f32, i32, P, P, P, P, P, i32, P, i32, i32, i32,
        P, P, P, P, P]
    lib.oracle_prepare_next_block.restype = ctypes.c_int64
    lib.oracle_stochastic_accept.argtypes = [P, P, P, P, i32, i32, i64, P, P,
                                             P, P, P, P, P, P, P, i32]
    lib.oracle_stochastic_accept.restype = ctypes.c_int
    lib.oracle_dflash2_select.argtypes = [P, P, P, P, P, P, i32, i32, i64,
                                          i32, i32, i32, i32, P, P, P, P, P,
                                          i32]
    lib.oracle_dflash2_select.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def decode_bf16(bits) -> np.ndarray:
    x = _c(bits, np.uint16).ravel()
    out = np.empty(x.size, np.float64)
    _load().oracle_decode_bf16(_ptr(x), x.size, _ptr(out))
    return out


def decode_fp16(bits) -> np.ndarray:
    x = _c(bits, np.uint16).ravel()
    out = np.empty(x.size, np.float64)
    _load().oracle_decode_fp16(_ptr(x), x.size, _ptr(out))
    return out


def decode_e4m3(bytes_) -> np.ndarray:
    x = _c(bytes_, np.uint8).ravel()
    out = np.empty(x.size, np.float64)
    _load().oracle_decode_e4m3(_ptr(x), x.size, _ptr(out))
    return out


def encode_fp16(x) -> np.ndarray:
    """float32 values -> fp16 bits, round-to-nearest-even."""
    a = _c(x, np.float32).ravel()
    out = np.empty(a.size, np.uint16)
    _load().oracle_encode_fp16(_ptr(a), a.size, _ptr(out))
    return out


def encode_e4m3(x) -> np.ndarray:
    """float32 values -> E4M3 bytes, round-to-nearest-even, saturated."""
    a = _c(x, np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    _load().oracle_encode_e4m3(_ptr(a), a.size, _ptr(out))
    return out


def kv_append(k_new_bits, v_new_bits, k_pages, v_pages, page_table, seq_lens,
              *, k_scales=None, v_scales=None, q_lens=None):
    """Block KV append on copies of the pool (q_lens: optional int32 [B] rows
    per request of a block padded to q_len).

    k_new_bits, v_new_bits: uint16 bf16 bits [B, q_len, Hkv, D]; pools as in
    verify_attention (uint8 + fp16-bit scales for FP8).  Returns
    (k_pages, v_pages, k_scales, v_scales, positions, cache_loc) with the
    pool arrays updated.
    """
    kn = _c(k_new_bits, np.uint16)
    vn = _c(v_new_bits, np.uint16)
    B, q_len, hkv, d = kn.shape
    fp8 = k_scales is not None
    kp = np.array(k_pages, dtype=np.uint8 if fp8 else np.uint16, copy=True)
    vp = np.array(v_pages, dtype=np.uint8 if fp8 else np.uint16, copy=True)
    ks = np.array(k_scales, dtype=np.uint16, copy=True) if fp8 else None
    vs = np.array(v_scales, dtype=np.uint16, copy=True) if fp8 else None
    num_pages, hkv2, page_size, _ = kp.shape
    assert hkv2 == hkv
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = None if q_lens is None else _c(q_lens, np.int32)
    pos = np.zeros((B, q_len), np.int32)
    loc = np.zeros((B, q_len), np.int64)
    rc = _load().oracle_kv_append(
        B, q_len, hkv, d, page_size, num_pages, pt.shape[1], int(fp8),
        _ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(pt),
        _ptr(sl), _ptr(ql), _ptr(pos), _ptr(loc))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle_kv_append failed with code {rc}")
    return kp, vp, ks, vs, pos, loc


def verify_attention(q_bits, k_pages, v_pages, page_table, seq_lens, *,
                     num_kv_heads: int, scale: float, k_scales=None,
                     v_scales=None, rows=None, key_begin: int = 0,
                     key_end: int = -1, threads: int = 0,
                     return_lse: bool = False, q_lens=None):
    """Verify attention in float64.

    q_bits:   uint16 bf16 bits [B, q_len, Hq, D]
    k_pages, v_pages: uint16 bf16 bits, or uint8 E4M3 bytes when scales are
              given, [num_pages, Hkv, page_size, D]
    k_scales, v_scales: uint16 fp16 bits [num_pages, Hkv, page_size, D/64]
    page_table: int32 [B, max_pages];  seq_lens: int32 [B] (block included)
    rows:     optional flat row ids (b*q_len + i)*Hq + h; default every row.
    q_lens:   optional int32 [B] rows per request (block padded to q_len);
              rows i >= q_lens[b] are zero.
    Returns out float64 [n_rows, D] (and lse [n_rows] if requested).
    """
    q = _c(q_bits, np.uint16)
    B, q_len, hq, d = q.shape
    fp8 = k_scales is not None
    kv_dtype = np.uint8 if fp8 else np.uint16
    kp = _c(k_pages, kv_dtype)
    vp = _c(v_pages, kv_dtype)
    num_pages, hkv, page_size, d2 = kp.shape
    assert d2 == d and hkv == num_kv_heads and vp.shape == kp.shape
    ks = _c(k_scales, np.uint16) if fp8 else None
    vs = _c(v_scales, np.uint16) if fp8 else None
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    assert pt.ndim == 2 and pt.shape[0] == B and sl.shape == (B,)
    ql = None if q_lens is None else _c(q_lens, np.int32)
    assert ql is None or ql.shape == (B,)
    r = None if rows is None else _c(rows, np.int64).ravel()
    n = B * q_len * hq if r is None else r.size
    out = np.zeros((n, d), np.float64)
    lse = np.zeros(n, np.float64)
    rc = _load().oracle_verify_attention(
        B, q_len, hq, hkv, d, page_size, num_pages, pt.shape[1], int(fp8),
        _ptr(q), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(pt), _ptr(sl),
        _ptr(ql), float(scale), _ptr(r), n, int(key_begin), int(key_end), _ptr(out),
        _ptr(lse), int(threads or default_threads()))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle_verify_attention failed with code {rc}")
    return (out, lse) if return_lse else out


def lse_merge(lse_parts, o_parts):
    """Merge split partials: lse [S], o [S, D] -> (out [D], lse)."""
    lse = _c(lse_parts, np.float64).ravel()
    o = _c(o_parts, np.float64)
    S, d = o.shape
    assert lse.size == S
    out = np.zeros(d, np.float64)
    lse_out = np.zeros(1, np.float64)
    _load().oracle_lse_merge(S, d, _ptr(lse), _ptr(o), _ptr(out), _ptr(lse_out))
    return out, float(lse_out[0])


def greedy_accept(logits, draft_ids, *, q_lens=None, seq_lens=None,
                  threads: int = 0):
    """Greedy acceptance.  logits fp32 [B*q_len, V]; draft_ids int32 [B, q_len];
    q_lens optional int32 [B] rows per request; seq_lens optional int32 [B].

    Returns dict with accept_len [B], next_token [B], out_tokens [B, q_len],
    argmax [B*q_len] and, when seq_lens is given, new_seq_lens [B].
    """
    lg = _c(logits, np.float32)
    dr = _c(draft_ids, np.int32)
    B, q_len = dr.shape
    assert lg.ndim == 2 and lg.shape[0] == B * q_len
    vocab = lg.shape[1]
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    toks = np.zeros((B, q_len), np.int32)
    am = np.zeros(B * q_len, np.int32)
    ql = None if q_lens is None else _c(q_lens, np.int32)
    sl = None if seq_lens is None else _c(seq_lens, np.int32)
    nsl = None if sl is None else np.zeros(B, np.int32)
    rc = _load().oracle_greedy_accept(
        _ptr(lg), _ptr(dr), _ptr(ql), B, q_len, vocab, _ptr(sl), _ptr(nsl),
        _ptr(acc), _ptr(nxt), _ptr(toks), _ptr(am),
        int(threads or default_threads()))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle_greedy_accept failed with code {rc}")
    res = {"accept_len": acc, "next_token": nxt, "out_tokens": toks,
           "argmax": am}
    if nsl is not None:
        res["new_seq_lens"] = nsl
    return res


WIDTH_POLICIES = {"fixed": 0, "ewma": 1, "doubling": 2}


def prepare_next_block(policy: str, q_max: int, q_lens, accept_len,
                       next_token, new_seq_lens, state, page_table, *,
                       page_size: int, num_pages: int, mask_id: int = 0,
                       min_width: int = 2, alpha: float = 0.5,
                       offset: float = 1.5):
    """Next verify width per request and the next block's layout.

    state: float32 [B] policy state (EWMA value or K), updated on a copy.
    Returns dict with next_q_lens, next_seq_lens [B]; block_ids, positions
    [B, q_max] int32; cache_loc [B, q_max] int64; state [B]; missing (rows
    without a reserved slot).
    """
    ql = _c(q_lens, np.int32)
    B = ql.shape[0]
    acc = _c(accept_len, np.int32)
    nxt = _c(next_token, np.int32)
    nsl = _c(new_seq_lens, np.int32)
    st = np.array(state, dtype=np.float32, copy=True)
    pt = _c(page_table, np.int32)
    out = {"next_q_lens": np.zeros(B, np.int32),
           "next_seq_lens": np.zeros(B, np.int32),
           "block_ids": np.zeros((B, q_max), np.int32),
           "positions": np.zeros((B, q_max), np.int32),
           "cache_loc": np.zeros((B, q_max), np.int64)}
    n = _load().oracle_prepare_next_block(
        WIDTH_POLICIES[policy], q_max, min_width, float(alpha), float(offset),
        B, _ptr(ql), _ptr(acc), _ptr(nxt), _ptr(nsl), _ptr(st), mask_id,
        _ptr(pt), pt.shape[1], page_size, num_pages, _ptr(out["next_q_lens"]),
        _ptr(out["next_seq_lens"]), _ptr(out["block_ids"]),
        _ptr(out["positions"]), _ptr(out["cache_loc"]))
    if n < 0:
        raise ValueError(f"oracle_prepare_next_block failed with code {n}")
    out["state"] = st
    out["missing"] = int(n)
    return out


def stochastic_accept(logits, draft_ids, temperature, u_accept, u_sample, *,
                      draft_probs=None, q_lens=None, seq_lens=None,
                      threads: int = 0):
    """Rejection-sampling verify in float64.

    logits fp32 [B*q_len, V]; draft_ids int32 [B, q_len]; temperature fp32
    [B] (> 0); u_accept fp32 [B, q_len-1] and u_sample fp32 [B] uniforms in
    [0, 1); draft_probs fp32 [B, q_len-1, V] or None (greedy drafts).
    Returns dict with accept_len, next_token, out_tokens, margin and, when
    seq_lens is given, new_seq_lens.
    """
    lg = _c(logits, np.float32)
    dr = _c(draft_ids, np.int32)
    B, q_len = dr.shape
    vocab = lg.shape[1]
    assert lg.shape[0] == B * q_len
    dp = None if draft_probs is None else _c(draft_probs, np.float32)
    assert dp is None or dp.shape == (B, q_len - 1, vocab)
    ql = None if q_lens is None else _c(q_lens, np.int32)
    tt = _c(temperature, np.float32).reshape(B)
    ua = _c(u_accept, np.float32).reshape(B, max(q_len - 1, 0))
    us = _c(u_sample, np.float32).reshape(B)
    sl = None if seq_lens is None else _c(seq_lens, np.int32)
    nsl = None if sl is None else np.zeros(B, np.int32)
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    toks = np.zeros((B, q_len), np.int32)
    mg = np.zeros(B, np.float64)
    rc = _load().oracle_stochastic_accept(
        _ptr(lg), _ptr(dr), _ptr(dp), _ptr(ql), B, q_len, vocab, _ptr(tt),
        _ptr(ua), _ptr(us), _ptr(sl), _ptr(nsl), _ptr(acc), _ptr(nxt),
        _ptr(toks), _ptr(mg), int(threads or default_threads()))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle_stochastic_accept failed with code {rc}")
    res = {"accept_len": acc, "next_token": nxt, "out_tokens": toks,
           "margin": mg}
    if nsl is not None:
        res["new_seq_lens"] = nsl
    return res


SELECT_MODES = {"greedy": 0, "map": 1}


def dflash2_select(cand_logits, boundary, hidden_bits, w_h_bits, code_a_bits,
                   code_b_bits, *, top: int = 16, mode: str = "greedy",
                   threads: int = 0):
    """DFlash2 candidate selection in float64.

    cand_logits fp32 [B, P-1, V]; boundary int32 [B]; hidden_bits bf16 bits
    [B, P-1, D]; w_h_bits [R, D]; code_a_bits, code_b_bits [V, R].
    Returns dict: cand_ids [B, P-1, K], cand_logit [B, P-1, K], trans
    [B, P-1, K, K], draft_ids [B, P], margin [B].
    """
    cl = _c(cand_logits, np.float32)
    B, P1, V = cl.shape
    bd = _c(boundary, np.int32).reshape(B)
    hb = _c(hidden_bits, np.uint16)
    D = hb.shape[2]
    assert hb.shape == (B, P1, D)
    wh = _c(w_h_bits, np.uint16)
    R = wh.shape[0]
    assert wh.shape == (R, D)
    ca = _c(code_a_bits, np.uint16)
    cb = _c(code_b_bits, np.uint16)
    assert ca.shape == (V, R) and cb.shape == (V, R)
    out = {"cand_ids": np.zeros((B, P1, top), np.int32),
           "cand_logit": np.zeros((B, P1, top), np.float64),
           "trans": np.zeros((B, P1, top, top), np.float64),
           "draft_ids": np.zeros((B, P1 + 1), np.int32),
           "margin": np.zeros(B, np.float64)}
    rc = _load().oracle_dflash2_select(
        _ptr(cl), _ptr(bd), _ptr(hb), _ptr(wh), _ptr(ca), _ptr(cb), B,
        P1 + 1, V, top, R, D, SELECT_MODES[mode], _ptr(out["cand_ids"]),
        _ptr(out["cand_logit"]), _ptr(out["trans"]), _ptr(out["draft_ids"]),
        _ptr(out["margin"]), int(threads or default_threads()))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle_dflash2_select failed with code {rc}")
    return out
