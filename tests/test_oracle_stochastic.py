"""Pins for the oracle's stochastic (rejection-sampling) verify (no GPU).

Hand-worked cases fix the accept ratio, the residual and the inverse-CDF
draw; Monte Carlo over drafts drawn from q checks the defining property of
speculative sampling (the committed tokens follow the target distribution)
and its acceptance rate sum_x min(p(x), q(x)); the zero-temperature limit
reduces to greedy acceptance."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle


def _run(p_rows, drafts, u_acc, u_s, q_rows=None, T=1.0, **kw):
    """One request per call row; p_rows [B, q_len, V] probabilities turned
    into logits by log (temperature 1 recovers them)."""
    p_rows = np.asarray(p_rows, np.float64)
    B, q_len, V = p_rows.shape
    with np.errstate(divide="ignore"):
        logits = (np.log(p_rows) * T).astype(np.float32).reshape(B * q_len, V)
    return oracle.stochastic_accept(
        logits, np.asarray(drafts, np.int32).reshape(B, q_len),
        np.full(B, T, np.float32), np.asarray(u_acc, np.float32).reshape(B, -1),
        np.asarray(u_s, np.float32).reshape(B),
        draft_probs=None if q_rows is None else
        np.asarray(q_rows, np.float32).reshape(B, q_len - 1, V), **kw)


def test_accept_ratio_and_residual_by_hand():
    p = [[[0.5, 0.3, 0.2], [0.1, 0.1, 0.8]]] * 3
    q = [[[0.2, 0.5, 0.3]]] * 3
    # d1 = 1: accept iff u < p/q = 0.6; residual max(0, p - q) = [0.3, 0, 0]
    r = _run(p, [[9, 1]] * 3, [[0.59], [0.61], [0.99]], [0.9, 0.0, 0.999],
             q_rows=q)
    assert r["accept_len"].tolist() == [1, 0, 0]
    # accepted: bonus from row 1 ([0.1, 0.1, 0.8], u = 0.9 -> index 2)
    assert r["next_token"].tolist() == [2, 0, 0]
    assert r["out_tokens"].tolist() == [[1, 2], [0, -1], [0, -1]]


def test_inverse_cdf_draw_by_hand():
    p = [[[0.25, 0.25, 0.5]]] * 4
    r = _run(p, [[0]] * 4, np.zeros((4, 0)), [0.1, 0.3, 0.6, 0.2499])
    assert r["accept_len"].tolist() == [0] * 4
    assert r["next_token"].tolist() == [0, 1, 2, 0]


def test_greedy_draft_residual_drops_the_draft_token():
    # one-hot q at d1 = 1: accept iff u < p(1) = 0.3; else draw from p
    # without token 1, renormalised to [5/7, 0, 2/7]
    p = [[[0.5, 0.3, 0.2], [0.2, 0.2, 0.6]]] * 3
    r = _run(p, [[4, 1]] * 3, [[0.29], [0.31], [0.31]], [0.0, 0.70, 0.72])
    assert r["accept_len"].tolist() == [1, 0, 0]
    assert r["next_token"].tolist() == [0, 0, 2]


def test_draft_equal_to_target_is_always_accepted():
    rng = np.random.default_rng(0)
    B, q_len, V = 50, 5, 7
    p = rng.dirichlet(np.ones(V), size=(B, q_len))
    drafts = rng.integers(0, V, (B, q_len))
    r = _run(p, drafts, rng.random((B, q_len - 1)) * 0.999, rng.random(B),
             q_rows=p[:, :-1])
    assert np.all(r["accept_len"] == q_len - 1)


def test_low_temperature_reduces_to_greedy():
    rng = np.random.default_rng(1)
    B, q_len, V = 64, 6, 40
    logits = rng.normal(size=(B * q_len, V)).astype(np.float32) * 3
    am = logits.argmax(1).reshape(B, q_len)
    drafts = rng.integers(0, V, (B, q_len)).astype(np.int32)
    hit = rng.random((B, q_len)) < 0.7
    drafts[:, 1:] = np.where(hit[:, 1:], am[:, :-1], drafts[:, 1:])
    g = oracle.greedy_accept(logits, drafts)
    s = oracle.stochastic_accept(logits, drafts, np.full(B, 1e-4, np.float32),
                                 rng.random((B, q_len - 1)).astype(np.float32),
                                 rng.random(B).astype(np.float32))
    assert np.array_equal(s["accept_len"], g["accept_len"])
    assert np.array_equal(s["next_token"], g["next_token"])


@pytest.mark.parametrize("T,greedy_draft", [(1.0, False), (0.7, False),
                                            (1.3, True)])
def test_committed_tokens_follow_the_target_distribution(T, greedy_draft):
    """Drafts drawn from q and target rows p: the first committed token is
    distributed as p_0, the second (given d1 was accepted) as p_1, and d1
    is accepted with probability sum_x min(p_0(x), q_1(x))."""
    rng = np.random.default_rng(int(T * 10) + greedy_draft)
    V, q_len, N = 6, 3, 200_000
    logits_rows = rng.normal(size=(q_len, V)) * 1.5
    p = softmax(logits_rows / T, axis=1)
    if greedy_draft:        # the drafter always proposes its own argmax
        q1 = np.eye(V)[rng.integers(0, V)]
        q2 = np.eye(V)[rng.integers(0, V)]
    else:
        q1, q2 = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    d1 = rng.choice(V, size=N, p=q1)
    d2 = rng.choice(V, size=N, p=q2)
    drafts = np.stack([np.zeros(N, int), d1, d2], 1)
    logits = np.tile(logits_rows.astype(np.float32), (N, 1))
    qp = None if greedy_draft else np.tile(np.stack([q1, q2]), (N, 1, 1))
    r = oracle.stochastic_accept(
        logits, drafts, np.full(N, T, np.float32),
        rng.random((N, 2)).astype(np.float32),
        rng.random(N).astype(np.float32), draft_probs=qp)
    t1 = r["out_tokens"][:, 0]
    freq1 = np.bincount(t1, minlength=V) / N
    tol = 5 * np.sqrt(p[0] * (1 - p[0]) / N) + 1e-4
    assert np.all(np.abs(freq1 - p[0]) < tol), (freq1, p[0])
    acc1 = (r["accept_len"] >= 1).mean()
    beta = np.minimum(p[0], q1).sum()
    assert abs(acc1 - beta) < 5 * np.sqrt(beta * (1 - beta) / N) + 1e-4
    sel = r["accept_len"] >= 1
    t2 = r["out_tokens"][sel, 1]
    n2 = sel.sum()
    freq2 = np.bincount(t2, minlength=V) / n2
    tol2 = 5 * np.sqrt(p[1] * (1 - p[1]) / n2) + 1e-4
    assert np.all(np.abs(freq2 - p[1]) < tol2), (freq2, p[1])


def test_ragged_rows_idle_requests_and_commit_lengths():
    rng = np.random.default_rng(3)
    B, q_max, V = 6, 5, 30
    logits = rng.normal(size=(B * q_max, V)).astype(np.float32)
    drafts = rng.integers(0, V, (B, q_max)).astype(np.int32)
    q_lens = np.array([5, 1, 0, 3, 2, 5], np.int32)
    seq = np.array([100, 50, 70, 9, 12, 1000], np.int32)
    ua = rng.random((B, q_max - 1)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    r = oracle.stochastic_accept(logits, drafts, np.ones(B, np.float32), ua,
                                 us, q_lens=q_lens, seq_lens=seq)
    assert r["accept_len"][2] == 0 and r["next_token"][2] == -1
    assert r["new_seq_lens"][2] == seq[2]
    assert np.all(r["accept_len"] <= np.maximum(q_lens - 1, 0))
    ok = q_lens > 0
    assert np.array_equal(r["new_seq_lens"][ok],
                          (seq - q_lens + r["accept_len"] + 1)[ok])
    # rows past q_b never matter: rewrite them and the result stays put
    lg2 = logits.reshape(B, q_max, V).copy()
    ua2 = ua.copy()
    for b in range(B):
        lg2[b, q_lens[b]:] = 7.0
        ua2[b, max(q_lens[b] - 1, 0):] = 0.0
    r2 = oracle.stochastic_accept(lg2.reshape(B * q_max, V), drafts,
                                  np.ones(B, np.float32), ua2, us,
                                  q_lens=q_lens, seq_lens=seq)
    for k in ("accept_len", "next_token", "out_tokens", "new_seq_lens"):
        assert np.array_equal(r[k], r2[k])


def test_zero_weight_tokens_are_never_drawn():
    # p = [0, 0.5, 0, 0.5]: even u = 0 must skip the zero-weight token 0
    p = [[[0.0, 0.5, 0.0, 0.5]]] * 3
    r = _run(p, [[0]] * 3, np.zeros((3, 0)), [0.0, 0.5, 0.9999])
    assert r["next_token"].tolist() == [1, 3, 3]
