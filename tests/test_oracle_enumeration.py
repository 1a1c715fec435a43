"""Exact-enumeration pins of the oracle (no GPU).

The pages state that accepting a proposal x ~ q with probability
min(1, p(x)/q(x)) makes the output distribution the anchor (AR) distribution
p (ai.arkapp.pw blog, ISD paragraph; de.news.hada.io, "Inference & ISD";
zhuanzhiai.com introduction: "provably matches").  These tests integrate the
oracle's decisions exactly over the 2^-24 uniform lattice and check that law:
the first emitted token is distributed as p for any q, and the first three
emitted tokens of a whole run follow the toy AR model's joint.
"""
import zlib
from collections import defaultdict

import numpy as np
import pytest

from isd_enum import forward_outcomes, softmax

NEG_INF = -np.inf
# lattice probabilities are exact multiples of 2^-24; a few factors multiply
TOL = 2e-6


def _first_token_law(prev_logits, logits, N, T, mode=0):
    """Law of the first token emitted by `logits` when the pending tokens were
    proposed (and their q saved) by the recovery forward `prev_logits`."""
    # the previous forward proposes x_1..x_{N-1} with q saved
    pend = defaultdict(float)
    for prob, _emit, newp, newq in forward_outcomes(prev_logits, None, None, None, N, T, mode=mode):
        pend[(newp, newq)] += prob
    assert abs(sum(pend.values()) - 1.0) < TOL
    law = defaultdict(float)
    for (p_tokens, q_vals), w in pend.items():
        for prob, emit, _np, _nq in forward_outcomes(logits, prev_logits if mode == 0 else None,
                                                     list(p_tokens), list(q_vals), N, T, mode=mode):
            law[emit[0]] += w * prob
    return law


def _rows(rng, N, V, scale=1.5):
    return (rng.standard_normal((2 * N - 1, V)) * scale).astype(np.float32)


CASES = ["random", "q_equals_p", "disjoint", "q_one_hot", "p_sparse_q_uniform", "q_wide"]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("N,V,T", [(2, 6, 1.0), (2, 5, 0.7), (3, 4, 1.3)])
def test_first_emitted_token_follows_anchor(case, N, V, T):
    rng = np.random.default_rng(zlib.crc32(repr((case, N, V)).encode()))
    prev = _rows(rng, N, V)
    cur = _rows(rng, N, V)
    q_row = N  # the previous forward's MASK row that proposed x_1
    if case == "q_equals_p":
        prev[q_row] = cur[0]
    elif case == "disjoint":
        half = V // 2
        cur[0, :half] = NEG_INF
        prev[q_row, half:] = NEG_INF
    elif case == "q_one_hot":
        prev[q_row, :] = NEG_INF
        prev[q_row, V - 1] = 0.0
    elif case == "p_sparse_q_uniform":
        cur[0, 1::2] = NEG_INF
        prev[q_row, :] = 0.0
    elif case == "q_wide":
        prev[q_row] *= 0.1
        cur[0] *= 3.0
    law = _first_token_law(prev, cur, N, T)
    p = softmax(cur[0], T)
    got = np.array([law.get(y, 0.0) for y in range(V)])
    assert abs(got.sum() - 1.0) < TOL
    np.testing.assert_allclose(got, p, atol=TOL, rtol=0)
    if case == "disjoint":
        # q has no mass where p has any: every proposal is rejected
        for y in range(V // 2):
            assert law.get(y, 0.0) == 0.0


def _toy_model(seed, V, scale, sparse=False):
    cache = {}

    def f(prefix):
        key = tuple(prefix)
        if key not in cache:
            h = zlib.crc32(repr((seed, key)).encode())
            row = (np.random.default_rng(h).standard_normal(V) * scale).astype(np.float32)
            if sparse and len(key) % 2 == 1:
                row[0] = NEG_INF
            cache[key] = row
        return cache[key]

    return f


def _forward_logits(f, g, prefix, pending, N, V):
    """Rows of one forward for a causal model f (anchors) and a proposal model g."""
    R = 2 * N - 1
    rows = np.zeros((R, V), dtype=np.float32)
    ctx = list(prefix) + (list(pending) if pending is not None else [])
    if pending is not None:
        for i in range(1, N):
            rows[i - 1] = f(list(prefix) + list(pending[:i - 1]))
    rows[N - 1] = f(ctx)
    for j in range(1, N):
        rows[N - 1 + j] = g(ctx + [-j])  # the j-th MASK position after ctx
    return rows


@pytest.mark.parametrize("N,V,T,sparse", [(2, 3, 1.0, False), (2, 3, 0.8, True), (3, 3, 1.0, False)])
def test_emitted_stream_follows_ar_joint(N, V, T, sparse):
    """Whole runs: the first three emitted tokens follow f's AR joint, whatever g is."""
    f = _toy_model(11, V, 1.2, sparse)
    g = _toy_model(23, V, 0.9)
    depth = 3
    law = defaultdict(float)

    def walk(prefix, pending, pq, prev_rows, prob):
        if len(prefix) >= depth:
            law[tuple(prefix[:depth])] += prob
            return
        rows = _forward_logits(f, g, prefix, pending, N, V)
        for p, emit, newp, newq in forward_outcomes(rows, prev_rows, pending, pq, N, T):
            walk(list(prefix) + list(emit), list(newp) if newp else None,
                 list(newq) if newq else None, rows, prob * p)

    walk([], None, None, None, 1.0)
    total = 0.0
    for path in np.ndindex(*([V] * depth)):
        expect = 1.0
        for t in range(depth):
            expect *= softmax(f(list(path[:t])), T)[path[t]]
        got = law.get(tuple(path), 0.0)
        assert abs(got - expect) < TOL, (path, got, expect)
        total += got
    assert abs(total - 1.0) < TOL



# Argmax proposals verified by sampling (mode 2): a proposal x is a point mass (q = 1), kept
# with probability p(x); after a rejection the replacement comes from max(0, p - delta_x),
# i.e. p without x.  The law of the emitted tokens is still p.
@pytest.mark.parametrize("case", ["random", "peaked_anchor", "proposal_unlikely", "masked"])
@pytest.mark.parametrize("N,V,T", [(2, 6, 1.0), (3, 4, 0.8)])
def test_argmax_proposals_first_token_follows_anchor(case, N, V, T):
    rng = np.random.default_rng(zlib.crc32(repr(("argmax", case, N, V)).encode()))
    prev = _rows(rng, N, V)
    cur = _rows(rng, N, V)
    x1 = int(np.argmax(prev[N]))  # the proposal the previous forward makes for position 1
    if case == "peaked_anchor":
        cur[0, x1] += 4.0
    elif case == "proposal_unlikely":
        cur[0, x1] -= 4.0
    elif case == "masked":
        cur[0, (x1 + 1) % V] = NEG_INF
    law = _first_token_law(prev, cur, N, T, mode=2)
    p = softmax(cur[0], T)
    got = np.array([law.get(y, 0.0) for y in range(V)])
    assert abs(got.sum() - 1.0) < TOL
    np.testing.assert_allclose(got, p, atol=TOL, rtol=0)


@pytest.mark.parametrize("N,V,T", [(2, 3, 1.0), (3, 3, 0.9)])
def test_argmax_proposals_stream_follows_ar_joint(N, V, T):
    f = _toy_model(31, V, 1.2)
    g = _toy_model(37, V, 0.9)
    depth = 3
    law = defaultdict(float)

    def walk(prefix, pending, pq, prob):
        if len(prefix) >= depth:
            law[tuple(prefix[:depth])] += prob
            return
        rows = _forward_logits(f, g, prefix, pending, N, V)
        for p, emit, newp, newq in forward_outcomes(rows, None, pending, pq, N, T, mode=2):
            walk(list(prefix) + list(emit), list(newp) if newp else None, list(newq) if newq else None,
                 prob * p)

    walk([], None, None, 1.0)
    for path in np.ndindex(*([V] * depth)):
        expect = 1.0
        for t in range(depth):
            expect *= softmax(f(list(path[:t])), T)[path[t]]
        assert abs(law.get(tuple(path), 0.0) - expect) < TOL, path
