"""The C-ABI library builds, loads and exports every declared symbol, and its
host-side argument checks reject bad calls before anything reaches a GPU
(no compute call is made here)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_target_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(spec_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert "spec_verify_attention" in declared
    assert "spec_greedy_accept" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(_native.EXPORTED) == set(declared)


def test_version_string(lib):
    assert b"sm_103a" in lib.spec_version()


def _desc(**kw):
    base = dict(batch=2, q_len=8, num_q_heads=24, num_kv_heads=4,
                head_dim=256, page_size=16, num_pages=64,
                max_pages_per_seq=8)
    base.update(kw)
    return _native.make_desc(**base)


FAKE = ctypes.c_void_p(0x100000)   # never dereferenced: checks come first


def _attn(lib, desc, q=FAKE, scale=0.0625, ws_bytes=1 << 30, out=FAKE,
          k_scales=None, v_scales=None):
    return lib.spec_verify_attention(
        ctypes.byref(desc) if desc is not None else None, q, FAKE, FAKE,
        k_scales, v_scales, FAKE, FAKE, scale, out, FAKE, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q_len=0), _native.SPEC_ERR_ARG),
    (dict(q_len=17), _native.SPEC_ERR_ARG),
    (dict(num_q_heads=25), _native.SPEC_ERR_ARG),
    (dict(num_kv_heads=0), _native.SPEC_ERR_ARG),
    (dict(head_dim=128), _native.SPEC_ERR_UNSUPPORTED),
    (dict(page_size=24), _native.SPEC_ERR_ARG),
    (dict(page_size=0), _native.SPEC_ERR_ARG),
    (dict(num_pages=0), _native.SPEC_ERR_ARG),
    (dict(batch=-1), _native.SPEC_ERR_ARG),
    (dict(batch=5000), _native.SPEC_ERR_ARG),
    (dict(q_len=16, num_q_heads=36, num_kv_heads=4), _native.SPEC_ERR_UNSUPPORTED),
])
def test_bad_descriptors_rejected(lib, kw, code):
    assert _attn(lib, _desc(**kw)) == code
    assert lib.spec_last_error()


def test_null_and_misaligned_pointers_rejected(lib):
    assert _attn(lib, None) == _native.SPEC_ERR_ARG
    assert _attn(lib, _desc(), q=None) == _native.SPEC_ERR_ARG
    assert _attn(lib, _desc(), q=ctypes.c_void_p(0x100008)) == \
        _native.SPEC_ERR_ALIGN
    assert _attn(lib, _desc(), out=ctypes.c_void_p(0x100002)) == \
        _native.SPEC_ERR_ALIGN
    assert _attn(lib, _desc(), scale=float("nan")) == _native.SPEC_ERR_ARG
    assert _attn(lib, _desc(), scale=float("inf")) == _native.SPEC_ERR_ARG
    assert _attn(lib, _desc(), scale=0.0) == _native.SPEC_ERR_ARG
    assert _attn(lib, _desc(), scale=-0.5) == _native.SPEC_ERR_ARG
    fp8 = _desc(kv_dtype="fp8")
    assert _attn(lib, fp8) == _native.SPEC_ERR_ARG          # scales missing
    assert _attn(lib, fp8, k_scales=ctypes.c_void_p(0x100008),
                 v_scales=FAKE) == _native.SPEC_ERR_ALIGN  # 16 B needed
    assert _attn(lib, _desc(kv_dtype="fp8", page_size=4), k_scales=FAKE,
                 v_scales=FAKE) == _native.SPEC_ERR_UNSUPPORTED


def test_empty_batch_is_a_noop(lib):
    assert _attn(lib, _desc(batch=0), q=None) == _native.SPEC_OK


def test_accept_argument_checks(lib):
    f = lib.spec_greedy_accept
    ok = dict(batch=2, q_len=8, vocab=1000)

    def call(batch=2, q_len=8, vocab=1000, logits=FAKE, ws=FAKE,
             ws_bytes=1 << 20, drafts=FAKE):
        return f(logits, drafts, batch, q_len, vocab, FAKE, FAKE, None, ws,
                 ws_bytes, None)

    assert call(q_len=0) == _native.SPEC_ERR_ARG
    assert call(q_len=17) == _native.SPEC_ERR_ARG
    assert call(vocab=0) == _native.SPEC_ERR_ARG
    assert call(batch=-3) == _native.SPEC_ERR_ARG
    assert call(batch=0, logits=None) == _native.SPEC_OK
    assert call(logits=None) == _native.SPEC_ERR_ARG
    assert call(drafts=ctypes.c_void_p(0x100001)) == _native.SPEC_ERR_ALIGN
    assert call(ws=None) == _native.SPEC_ERR_WORKSPACE
    need = lib.spec_accept_workspace_size(16, 1000)
    assert call(ws_bytes=need - 1) == _native.SPEC_ERR_WORKSPACE
    assert ok


def test_accept_workspace_size_formula(lib):
    # one (fp32 value, int32 index) pair per row and 8192-entry vocab
    # chunk, and one completion counter per row (at most one per request)
    chunks = -(-248320 // 8192)
    n = lib.spec_accept_workspace_size(64, 248320)
    assert n >= 64 * chunks * 8 + 64 * 4
    assert n <= 64 * chunks * 8 + 64 * 4 + 4 * 256
    assert lib.spec_accept_workspace_size(-1, 10) == 0


def test_kv_append_argument_checks(lib):
    def call(desc, k_new=FAKE, ks=None, vs=None, pos=None, loc=None, ws=None):
        return lib.spec_kv_append(
            ctypes.byref(desc) if desc is not None else None, k_new, FAKE,
            FAKE, FAKE, ks, vs, FAKE, FAKE, pos, loc, ws, None)

    assert call(None) == _native.SPEC_ERR_ARG
    assert call(_desc(batch=0), k_new=None) == _native.SPEC_OK
    assert call(_desc(), k_new=None) == _native.SPEC_ERR_ARG
    assert call(_desc(), k_new=ctypes.c_void_p(0x100008)) == \
        _native.SPEC_ERR_ALIGN
    assert call(_desc(), loc=ctypes.c_void_p(0x100004)) == \
        _native.SPEC_ERR_ALIGN
    assert call(_desc(kv_dtype="fp8")) == _native.SPEC_ERR_ARG
    assert call(_desc(kv_dtype="fp8"), ks=FAKE,
                vs=ctypes.c_void_p(0x100002)) == _native.SPEC_ERR_ALIGN
    assert call(_desc(checked=True)) == _native.SPEC_ERR_WORKSPACE
    assert call(_desc(page_size=24)) == _native.SPEC_ERR_ARG


def test_accept_commit_argument_checks(lib):
    f = lib.spec_greedy_accept_commit

    def call(q_lens=None, seq_lens=None, new=None):
        return f(FAKE, FAKE, q_lens, 2, 8, 1000, seq_lens, new, FAKE, FAKE,
                 None, FAKE, 1 << 20, None)

    assert call(seq_lens=FAKE) == _native.SPEC_ERR_ARG      # needs new too
    assert call(new=FAKE) == _native.SPEC_ERR_ARG
    assert call(q_lens=ctypes.c_void_p(0x100002)) == _native.SPEC_ERR_ALIGN
    assert call(seq_lens=FAKE, new=ctypes.c_void_p(0x100001)) == \
        _native.SPEC_ERR_ALIGN


def test_desc_q_lens_must_be_aligned(lib):
    d = _desc()
    d.q_lens = 0x100002
    assert _attn(lib, d) == _native.SPEC_ERR_ALIGN


def test_prepare_next_block_argument_checks(lib):
    f = lib.spec_prepare_next_block

    def call(pol, batch=3, state=FAKE, cache_loc=FAKE, next_q=FAKE):
        return f(ctypes.byref(pol) if pol is not None else None, batch, None,
                 FAKE, FAKE, FAKE, state, FAKE, 4, 16, 64, next_q, FAKE, FAKE,
                 FAKE, cache_loc, None, None)

    ok = _native.width_policy("ewma", 8)
    assert call(None) == _native.SPEC_ERR_ARG
    assert call(_native.width_policy("fixed", 17)) == _native.SPEC_ERR_ARG
    assert call(_native.width_policy("ewma", 8, min_width=9)) == \
        _native.SPEC_ERR_ARG
    assert call(_native.width_policy("ewma", 8, alpha=1.5)) == \
        _native.SPEC_ERR_ARG
    assert call(_native.width_policy("ewma", 8, offset=float("nan"))) == \
        _native.SPEC_ERR_ARG
    bad = _native.width_policy("fixed", 8)
    bad.policy = 3
    assert call(bad) == _native.SPEC_ERR_ARG
    assert call(ok, state=None) == _native.SPEC_ERR_ARG
    assert call(_native.width_policy("fixed", 8), batch=0, state=None,
                next_q=None) == _native.SPEC_OK
    assert call(ok, next_q=None) == _native.SPEC_ERR_ARG
    assert call(ok, cache_loc=ctypes.c_void_p(0x100004)) == \
        _native.SPEC_ERR_ALIGN
    assert call(ok, batch=-1) == _native.SPEC_ERR_ARG


def test_stochastic_accept_argument_checks(lib):
    f = lib.spec_stochastic_accept

    def call(q_len=8, u_accept=FAKE, seq=None, new=None, temp=FAKE,
             ws_bytes=1 << 24, ws=FAKE, probs=None):
        return f(FAKE, FAKE, probs, None, 2, q_len, 1000, temp, u_accept,
                 FAKE, seq, new, FAKE, FAKE, None, ws, ws_bytes, None)

    assert call(q_len=0) == _native.SPEC_ERR_ARG
    assert call(q_len=17) == _native.SPEC_ERR_ARG
    assert call(u_accept=None) == _native.SPEC_ERR_ARG
    assert call(temp=None) == _native.SPEC_ERR_ARG
    assert call(seq=FAKE) == _native.SPEC_ERR_ARG
    assert call(probs=ctypes.c_void_p(0x100002)) == _native.SPEC_ERR_ALIGN
    assert call(ws=None) == _native.SPEC_ERR_WORKSPACE
    need = lib.spec_stochastic_workspace_size(2, 8, 1000)
    assert need > 0
    assert call(ws_bytes=need - 1) == _native.SPEC_ERR_WORKSPACE
    assert lib.spec_stochastic_workspace_size(2, 0, 1000) == 0


def test_select_argument_checks(lib):
    def d(**kw):
        base = dict(batch=2, positions=8, vocab=248320, top=16, rank=256,
                    dim=5120, mode=0)
        base.update(kw)
        return _native.SelectDesc(*base.values())

    size = lib.spec_select_workspace_size
    assert size(ctypes.byref(d())) > 0
    for bad in (dict(positions=1), dict(positions=17), dict(top=0),
                dict(top=17), dict(vocab=262145), dict(vocab=8, top=16),
                dict(rank=260), dict(rank=12), dict(dim=24), dict(mode=2),
                dict(batch=-1)):
        assert size(ctypes.byref(d(**bad))) == 0, bad
    f = lib.spec_dflash2_select

    def call(desc, logits=FAKE, ws=FAKE, ws_bytes=1 << 30, hidden=FAKE):
        return f(ctypes.byref(desc), logits, FAKE, hidden, FAKE, FAKE, FAKE,
                 FAKE, None, None, None, ws, ws_bytes, None)

    assert call(d(batch=0), logits=None) == _native.SPEC_OK
    assert call(d(), logits=None) == _native.SPEC_ERR_ARG
    assert call(d(), hidden=ctypes.c_void_p(0x100002)) == _native.SPEC_ERR_ALIGN
    assert call(d(), ws=None) == _native.SPEC_ERR_WORKSPACE
    assert call(d(), ws_bytes=16) == _native.SPEC_ERR_WORKSPACE


def test_wait_limit_hook_range(lib):
    # the checked-mode wait bound: [0, 4e9] cycles, 0 = the default
    assert lib.spec_verify_set_wait_limit(-1) == _native.SPEC_ERR_ARG
    assert lib.spec_verify_set_wait_limit(5_000_000_000) == _native.SPEC_ERR_ARG
    assert lib.spec_verify_set_wait_limit(1000) == _native.SPEC_OK
    assert lib.spec_verify_set_wait_limit(0) == _native.SPEC_OK
