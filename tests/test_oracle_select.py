"""Pins for the oracle's DFlash2 candidate selector (no GPU).

Top-K against numpy's lexsort; K = 1 and zero codebooks reduce both walks to
a per-position argmax; one-hot codebooks give the transition table in closed
form; the projection is linear; the MAP walk equals a brute force over every
path; a hand-worked case separates the greedy walk from the MAP walk."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_target_gb300 import workloads as wl


def _bits(x):
    return wl.to_numpy_bits(torch.as_tensor(np.asarray(x, np.float32)).to(
        torch.bfloat16))


def _rand(B=3, P=6, V=500, R=16, D=24, seed=0, scale=0.5):
    rng = np.random.default_rng(seed)
    return dict(
        cand_logits=(rng.normal(size=(B, P - 1, V)) * 2).astype(np.float32),
        boundary=rng.integers(0, V, B).astype(np.int32),
        hidden_bits=_bits(rng.normal(size=(B, P - 1, D))),
        w_h_bits=_bits(rng.normal(size=(R, D)) / np.sqrt(D)),
        code_a_bits=_bits(rng.normal(size=(V, R)) * scale),
        code_b_bits=_bits(rng.normal(size=(V, R)) * scale))


def test_top_k_matches_lexsort_with_ties_and_infinities():
    inp = _rand(B=2, P=4, V=300, seed=1)
    cl = inp["cand_logits"]
    cl[0, 0, [3, 50, 7, 299]] = 9.0          # a tie for the top
    cl[1, 1, :] = -np.inf
    cl[1, 1, [10, 20]] = [1.0, 1.0]            # fewer finite than K
    r = oracle.dflash2_select(**inp, top=8)
    for b in range(2):
        for t in range(3):
            x = cl[b, t]
            order = np.lexsort((np.arange(x.size), -x))[:8]
            assert np.array_equal(r["cand_ids"][b, t], order)
            assert np.array_equal(r["cand_logit"][b, t], x[order])


@pytest.mark.parametrize("mode", ["greedy", "map"])
def test_top1_and_zero_codebooks_reduce_to_argmax(mode):
    inp = _rand(seed=2)
    am = inp["cand_logits"].argmax(axis=2)
    r = oracle.dflash2_select(**inp, top=1, mode=mode)
    assert np.array_equal(r["draft_ids"][:, 1:], am)
    inp["code_a_bits"] = np.zeros_like(inp["code_a_bits"])
    r = oracle.dflash2_select(**inp, top=16, mode=mode)
    assert np.array_equal(r["draft_ids"][:, 1:], am)
    assert np.array_equal(r["draft_ids"][:, 0], inp["boundary"])


def test_one_hot_codebooks_give_the_closed_form():
    # A(a) = e_{a % R}, B(b) = e_{3b % R}, W_H a cyclic shift (D = R, so
    # H_t[r] = h_t[(r + 1) % R]): the interaction is h_t[(a % R + 1) % R]
    # when a % R == 3b % R, else 0.  Neither map is symmetric, so a
    # transposed projection or swapped codebooks change the table.
    B, P, V, R = 2, 4, 40, 8
    rng = np.random.default_rng(3)
    eye = np.eye(R)
    shift = np.roll(eye, 1, axis=1)            # shift[r, (r + 1) % R] = 1
    inp = dict(cand_logits=rng.normal(size=(B, P - 1, V)).astype(np.float32),
               boundary=np.array([5, 12], np.int32),
               hidden_bits=_bits(rng.integers(-4, 5, (B, P - 1, R))),
               w_h_bits=_bits(shift),
               code_a_bits=_bits(eye[np.arange(V) % R]),
               code_b_bits=_bits(eye[(3 * np.arange(V)) % R]))
    r = oracle.dflash2_select(**inp, top=6)
    hid = torch.from_numpy(inp["hidden_bits"].view(np.int16)).view(
        torch.bfloat16).double().numpy()
    hits = 0
    for b in range(B):
        for t in range(1, P):
            preds = [inp["boundary"][b]] if t == 1 else r["cand_ids"][b, t - 2]
            for ai, a in enumerate(preds):
                for ci, c in enumerate(r["cand_ids"][b, t - 1]):
                    want = float(inp["cand_logits"][b, t - 1, c])
                    if a % R == (3 * c) % R:
                        want += float(hid[b, t - 1, (a % R + 1) % R])
                        hits += 1
                    assert r["trans"][b, t - 1, ai, ci] == want
            if t == 1:
                assert np.all(r["trans"][b, 0, 1:] == -np.inf)
    assert hits > 5


def test_projection_is_linear():
    inp = _rand(seed=4)
    r1 = oracle.dflash2_select(**inp, top=5)
    w = torch.from_numpy(inp["w_h_bits"].view(np.int16)).view(torch.bfloat16)
    inp["w_h_bits"] = wl.to_numpy_bits(w * 2)          # exact in bf16
    r2 = oracle.dflash2_select(**inp, top=5)
    u = r1["cand_logit"][:, :, None, :]
    ok = np.isfinite(r1["trans"])
    # (U + x) - U rounds, so compare to the last few ulps of U
    np.testing.assert_allclose((r2["trans"] - u)[ok], 2 * (r1["trans"] - u)[ok],
                               rtol=1e-12, atol=1e-13)


def _path_score(trans, ids, path):
    s, prev = 0.0, 0
    for t, c in enumerate(path):
        s += trans[t, prev, c]
        prev = c
    return s


@pytest.mark.parametrize("seed", range(4))
def test_map_walk_equals_brute_force_and_beats_greedy(seed):
    K, P = 3, 5
    inp = _rand(B=4, P=P, V=60, seed=10 + seed, scale=1.5)
    g = oracle.dflash2_select(**inp, top=K, mode="greedy")
    m = oracle.dflash2_select(**inp, top=K, mode="map")
    assert np.array_equal(g["trans"], m["trans"])
    for b in range(4):
        tr = m["trans"][b]
        scores = {p: _path_score(tr, None, p)
                  for p in itertools.product(range(K), repeat=P - 1)}
        best = max(scores.values())
        # lowest-rank path among equal maxima: lexicographically from the end
        # back (the walk breaks ties at the final position, then backwards)
        chosen = [m["cand_ids"][b, t].tolist().index(m["draft_ids"][b, t + 1])
                  for t in range(P - 1)]
        assert scores[tuple(chosen)] == best
        gchosen = [g["cand_ids"][b, t].tolist().index(g["draft_ids"][b, t + 1])
                   for t in range(P - 1)]
        assert scores[tuple(gchosen)] <= best
        # the greedy walk takes the best successor of its own predecessor
        prev = 0
        for t, c in enumerate(gchosen):
            assert tr[t, prev, c] == tr[t, prev].max()
            prev = c


def test_greedy_and_map_differ_on_a_hand_worked_case():
    # K = 2, P = 3, R = D = 1, W_H = 1, h = 1.  Candidates at t = 1: token 0
    # (logit 1.0) and token 1 (logit 0.9); at t = 2: token 2 (0.0) and
    # token 3 (0.0).  A = 0 for the boundary, A(1) = 2, A(0) = 0;
    # B(3) = 2, others 0.
    #   greedy: t1 picks token 0 (1.0 > 0.9), t2 from token 0: both 0 ->
    #           rank 0 (token 2); chain score 1.0
    #   MAP:    token 1 then token 3 scores 0.9 + (0 + 2 * 1 * 2) = 4.9
    V = 6
    logits = np.full((1, 2, V), -10.0, np.float32)
    logits[0, 0, 0], logits[0, 0, 1] = 1.0, 0.9
    logits[0, 1, 2], logits[0, 1, 3] = 0.0, 0.0
    a = np.zeros((V, 1))
    a[1] = 2.0
    bb = np.zeros((V, 1))
    bb[3] = 2.0
    inp = dict(cand_logits=logits, boundary=np.array([5], np.int32),
               hidden_bits=_bits(np.ones((1, 2, 1))),
               w_h_bits=_bits(np.ones((1, 1))),
               code_a_bits=_bits(a), code_b_bits=_bits(bb))
    g = oracle.dflash2_select(**inp, top=2, mode="greedy")
    m = oracle.dflash2_select(**inp, top=2, mode="map")
    assert g["draft_ids"].tolist() == [[5, 0, 2]]
    assert m["draft_ids"].tolist() == [[5, 1, 3]]
    assert m["trans"][0, 1, 1, 1] == 4.0
    assert g["margin"][0] == 0.0                 # the tie at t = 2
