"""GPU stochastic verify (rejection sampling, through the C ABI) against the
oracle.  The kernels decide in float32 and the oracle in float64, so a
request may differ only where one of its decisions lies within rounding of
its threshold: every mismatch must have a small oracle margin, and such
requests must be rare.  A Monte Carlo run on the GPU checks the defining
property directly: committed tokens follow the target distribution."""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
import speculative_decoding_target_gb300 as sv
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"
MARGIN = 1e-4          # decisions closer than this to their threshold may flip


def _case(B, q_len, V, *, with_q, seed, ragged=True, T=(0.5, 1.5),
          accept_bias=0.6):
    rng = np.random.default_rng(seed)
    logits = (rng.normal(size=(B * q_len, V)) * 2).astype(np.float32)
    temp = rng.uniform(*T, size=B).astype(np.float32)
    p = softmax(logits.astype(np.float64).reshape(B, q_len, V) /
                temp[:, None, None], axis=2)
    drafts = np.zeros((B, q_len), np.int32)
    drafts[:, 0] = rng.integers(0, V, B)
    qp = None
    if with_q:   # a drafter near the target: mixtures of p and noise
        noise = rng.dirichlet(np.ones(min(V, 64)), size=(B, q_len - 1))
        qfull = np.zeros((B, q_len - 1, V))
        qfull[:, :, :noise.shape[2]] = noise
        q64 = accept_bias * p[:, :-1] + (1 - accept_bias) * qfull
        q64 /= q64.sum(2, keepdims=True)
        qp = q64.astype(np.float32)
        cdf = np.cumsum(q64, axis=2)
        for b in range(B):
            for j in range(1, q_len):
                c = cdf[b, j - 1]
                drafts[b, j] = min(int(np.searchsorted(
                    c, rng.random() * c[-1], side="right")), V - 1)
    else:        # greedy drafter: the target's argmax most of the time
        am = p.argmax(2)
        hit = rng.random((B, q_len)) < accept_bias
        drafts[:, 1:] = np.where(hit[:, 1:], am[:, :-1],
                                 rng.integers(0, V, (B, q_len - 1)))
    ql = (rng.integers(0, q_len + 1, B) if ragged else
          np.full(B, q_len)).astype(np.int32)
    ql[0] = q_len
    seq = rng.integers(q_len, 5000, B).astype(np.int32)
    ua = rng.random((B, q_len - 1)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    return dict(logits=logits, drafts=drafts, qp=qp, ql=ql, temp=temp,
                ua=ua, us=us, seq=seq)


def _compare(c, max_flip_frac=0.02):
    ensure_built()
    d = lambda a: None if a is None else torch.from_numpy(a).to(DEV)
    acc, nxt, toks, new = sv.stochastic_accept(
        d(c["logits"]), d(c["drafts"]), d(c["temp"]), d(c["ua"]),
        d(c["us"]), draft_probs=d(c["qp"]), q_lens=d(c["ql"]),
        seq_lens=d(c["seq"]))
    torch.cuda.synchronize()
    ref = oracle.stochastic_accept(
        c["logits"], c["drafts"], c["temp"], c["ua"], c["us"],
        draft_probs=c["qp"], q_lens=c["ql"], seq_lens=c["seq"])
    got = {"accept_len": acc, "next_token": nxt, "out_tokens": toks,
           "new_seq_lens": new}
    same = np.ones(len(c["ql"]), bool)
    for k, v in got.items():
        g = v.cpu().numpy()
        eq = g == ref[k]
        same &= eq if eq.ndim == 1 else eq.all(1)
    flips = np.flatnonzero(~same)
    assert np.all(ref["margin"][flips] < MARGIN), \
        (flips, ref["margin"][flips])
    assert len(flips) <= max(1, max_flip_frac * len(same))
    return ref, same


@pytest.mark.parametrize("with_q", [True, False])
@pytest.mark.parametrize("B,q_len,V", [(64, 8, 3000), (16, 16, 50000),
                                       (40, 4, 8193), (12, 2, 7)])
def test_matches_oracle(B, q_len, V, with_q):
    _compare(_case(B, q_len, V, with_q=with_q, seed=B + q_len + V + with_q))


def test_production_vocab_and_scalar_path():
    _compare(_case(8, 8, 248320, with_q=True, seed=1))
    _compare(_case(6, 8, 248319, with_q=False, seed=2))   # vocab % 4 != 0


def test_single_row_blocks_draw_the_bonus():
    c = _case(32, 1, 1000, with_q=False, seed=3, ragged=False)
    ref, _ = _compare(c)
    assert np.all(ref["accept_len"] == 0)


def test_committed_tokens_follow_the_target_distribution_on_gpu():
    ensure_built()
    rng = np.random.default_rng(11)
    V, q_len, n, T = 5, 2, 32000, 0.8      # two batches: rows <= 65535
    row = rng.normal(size=(q_len, V)) * 1.5
    p0 = softmax(row[0] / T)
    q1 = rng.dirichlet(np.ones(V))
    logits = np.tile(row.astype(np.float32), (n, 1))
    qp = np.tile(q1.astype(np.float32), (n, 1, 1))
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    t1, a1 = [], []
    for _ in range(2):
        drafts = np.stack([np.zeros(n, int), rng.choice(V, size=n, p=q1)],
                          1).astype(np.int32)
        acc, nxt, toks, _ = sv.stochastic_accept(
            d(logits), d(drafts), d(np.full(n, T, np.float32)),
            d(rng.random((n, 1)).astype(np.float32)),
            d(rng.random(n).astype(np.float32)), draft_probs=d(qp))
        t1.append(toks[:, 0].cpu().numpy())
        a1.append(acc.cpu().numpy())
    t1, a1 = np.concatenate(t1), np.concatenate(a1)
    N = t1.size
    freq = np.bincount(t1, minlength=V) / N
    tol = 5 * np.sqrt(p0 * (1 - p0) / N) + 1e-4
    assert np.all(np.abs(freq - p0) < tol), (freq, p0)
    beta = np.minimum(p0, q1).sum()
    a1 = (a1 >= 1).mean()
    assert abs(a1 - beta) < 5 * np.sqrt(beta * (1 - beta) / N) + 1e-4
