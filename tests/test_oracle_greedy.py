"""Greedy (argmax) mode of the oracle: the lossless invariant and special cases.

Argmax proposals are one of the serving optimisations the pages list (ai.arkapp.pw,
"實際部署"; de.news.hada.io, "Serving (SGLang)"), and the method is claimed to
match the AR model's output.  With greedy decisions everywhere, the emitted
stream must equal step-by-step argmax decoding of the anchor model, whatever
the proposals are.
"""
import zlib

import numpy as np
import pytest

import oracle


class ToyAR:
    """A deterministic causal 'model': logits = seeded function of the prefix."""

    def __init__(self, seed, V, scale=2.0):
        self.seed, self.V, self.scale, self.cache = seed, V, scale, {}

    def __call__(self, prefix):
        key = tuple(prefix)
        if key not in self.cache:
            h = zlib.crc32(repr((self.seed, key)).encode())
            self.cache[key] = (np.random.default_rng(h).standard_normal(self.V)
                               * self.scale).astype(np.float32)
        return self.cache[key]

    def greedy(self, prefix, n):
        out = list(prefix)
        for _ in range(n):
            out.append(int(np.argmax(self(out))))
        return out[len(prefix):]


def _forward_rows(f, prefix, pending, N, V, noise, rng):
    """Anchor rows from f; MASK rows guess f's greedy continuation after the
    bonus position, blurred by noise so that proposals are sometimes wrong."""
    R = 2 * N - 1
    rows = np.zeros((R, V), dtype=np.float32)
    ctx = list(prefix) + (list(pending) if pending is not None else [])
    if pending is not None:
        for i in range(1, N):
            rows[i - 1] = f(list(prefix) + list(pending[:i - 1]))
    rows[N - 1] = f(ctx)
    cont = f.greedy(ctx, N)  # bonus then N-1 more
    for j in range(1, N):
        rows[N - 1 + j] = f(ctx + cont[:j]) + noise * rng.standard_normal(V).astype(np.float32)
    return rows


def run_isd(f, N, V, n_tokens, noise, seed, greedy=True, T=1.0):
    rng = np.random.default_rng(seed)
    prefix, pending, pq, prev = [], None, None, None
    forwards = 0
    while len(prefix) < n_tokens:
        rows = _forward_rows(f, prefix, pending, N, V, noise, rng)
        pt = np.array([pending if pending else [-1] * (N - 1)], dtype=np.int32)
        q = np.array([pq if pq else [0.0] * (N - 1)], dtype=np.float32)
        res = oracle.isd_step(rows[None], None if prev is None else prev[None], pt, q, N, T,
                              greedy, seed, forwards, dtype="f32")
        assert res["seq_status"][0] == 0
        n = int(res["accepted_len"][0])
        prefix += [int(t) for t in res["tokens_out"][0, :n]]
        newp = res["tokens_out"][0, N:]
        pending = [int(t) for t in newp] if newp[0] >= 0 else None
        pq = [float(x) for x in res["new_q"][0]] if pending else None
        prev = rows
        forwards += 1
    return prefix[:n_tokens], forwards


@pytest.mark.parametrize("N", [2, 3, 4, 8])
@pytest.mark.parametrize("noise", [0.0, 0.8, 3.0])
def test_greedy_stream_equals_ar_argmax(N, noise):
    V = 40
    f = ToyAR(5 + N, V)
    n = 60
    stream, forwards = run_isd(f, N, V, n, noise, seed=N * 10 + int(noise * 10))
    assert stream == f.greedy([], n)
    if noise == 0.0:
        # perfect proposals: every forward after the first emits N tokens
        assert forwards == 1 + int(np.ceil((n - 1) / N))


def test_greedy_argmax_ties_take_lowest_index():
    N, V = 2, 6
    rows = np.zeros((1, 3, V), dtype=np.float32)
    rows[0, 1, [2, 4]] = 5.0  # tie between tokens 2 and 4 in the anchor row
    rows[0, 2, [1, 3]] = 7.0
    res = oracle.isd_step(rows, None, [[-1]], [[0.0]], N, 1.0, True, 0, 0, dtype="f32")
    assert res["tokens_out"][0].tolist() == [2, -1, 1]
    assert res["new_q"][0, 0] == 1.0


def test_low_temperature_sampling_equals_greedy():
    """T -> 0: softmax concentrates on the argmax; the sampled run equals greedy."""
    V = 30
    f = ToyAR(77, V, scale=3.0)
    s_greedy, _ = run_isd(f, 4, V, 40, 1.0, seed=3, greedy=True)
    s_cold, _ = run_isd(f, 4, V, 40, 1.0, seed=3, greedy=False, T=1e-4)
    assert s_cold == s_greedy


def test_p_equals_q_accepts_everything():
    """Identical anchor and proposal rows: min(1, p/q) = 1, so N tokens per forward."""
    N, V, B = 4, 50, 16
    rng = np.random.default_rng(9)
    rows = rng.standard_normal((B, 2 * N - 1, V)).astype(np.float32)
    pending = -np.ones((B, N - 1), dtype=np.int32)
    pq = np.zeros((B, N - 1), dtype=np.float32)
    prev = None
    for t in range(30):
        cur = rng.standard_normal((B, 2 * N - 1, V)).astype(np.float32)
        if prev is not None:
            cur[:, :N - 1] = prev[:, N:]  # anchor row i-1 = MASK row that proposed x_i
        res = oracle.isd_step(cur, prev, pending, pq, N, 1.0, False, 4, t, dtype="f32")
        if t > 0:
            assert (res["accepted_len"] == N).all()
        pending = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)
        prev = cur


def test_disjoint_support_always_rejects_first():
    """q puts no mass where p has any: K=0 every time, the replacement comes from p."""
    N, V, B = 3, 10, 64
    rng = np.random.default_rng(2)
    counts = np.zeros(V)
    pending = -np.ones((B, N - 1), dtype=np.int32)
    pq = np.zeros((B, N - 1), dtype=np.float32)
    prev = None
    anchor = rng.standard_normal(V).astype(np.float32)
    anchor[5:] = -np.inf
    for t in range(200):
        cur = rng.standard_normal((B, 2 * N - 1, V)).astype(np.float32)
        cur[:, N:, :5] = -np.inf  # proposals only among tokens 5..9
        cur[:, :N - 1] = anchor  # anchors only among tokens 0..4
        res = oracle.isd_step(cur, prev, pending, pq, N, 1.0, False, 8, t, dtype="f32")
        had = pending[:, 0] >= 0
        assert (res["accepted_len"][had] == 1).all()
        assert (res["tokens_out"][had, N] == -1).all()
        for y in res["tokens_out"][had, 0]:
            counts[y] += 1
        pending = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)
        prev = cur
    p = np.exp(anchor.astype(np.float64) - anchor[:5].max())
    p[5:] = 0
    p /= p.sum()
    n = counts.sum()
    assert n > 3000
    assert counts[5:].sum() == 0
    # chi-square goodness of fit, 4 degrees of freedom, ~0.1% level
    chi2 = ((counts[:5] - n * p[:5]) ** 2 / (n * p[:5])).sum()
    assert chi2 < 18.5


def test_single_token_vocabulary():
    N, V, B = 3, 1, 4
    rows = np.zeros((B, 2 * N - 1, V), dtype=np.float32)
    pending = -np.ones((B, N - 1), dtype=np.int32)
    pq = np.zeros((B, N - 1), dtype=np.float32)
    for t in range(3):
        for greedy in (False, True):
            res = oracle.isd_step(rows, rows, pending, pq, N, 1.0, greedy, 0, t, dtype="f32")
            assert (res["tokens_out"][:, :int(res["accepted_len"][0])] == 0).all()
            assert (res["new_q"] == 1.0).all()
        assert (res["accepted_len"] == (1 if t == 0 else N)).all()
        pending = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)


def test_bad_inputs_flag_the_sequence():
    N, V = 2, 8
    rows = np.zeros((3, 3, V), dtype=np.float32)
    rows[1, 0, 3] = np.nan   # seq 1 has pending tokens: row 0 is read
    rows[2, 0, 3] = np.nan   # seq 2 is recovering: row 0 is not read
    pending = np.array([[1], [1], [-1]], dtype=np.int32)
    pq = np.array([[0.5], [0.5], [0.0]], dtype=np.float32)
    res = oracle.isd_step(rows, rows, pending, pq, N, 1.0, False, 0, 0, dtype="f32")
    assert res["seq_status"].tolist() == [0, oracle.SEQ_NONFINITE, 0]
    assert res["accepted_len"][1] == 0 and (res["tokens_out"][1] == -1).all()
    res = oracle.isd_step(rows[:1], rows[:1], [[V]], [[0.5]], N, 1.0, False, 0, 0, dtype="f32")
    assert res["seq_status"][0] == oracle.SEQ_BAD_PENDING
    res = oracle.isd_step(rows[:1], rows[:1], [[2]], [[0.0]], N, 1.0, False, 0, 0, dtype="f32")
    assert res["seq_status"][0] == oracle.SEQ_BAD_PENDING
    allneg = np.full((1, 3, V), -np.inf, dtype=np.float32)
    res = oracle.isd_step(allneg, None, [[-1]], [[0.0]], N, 1.0, False, 0, 0, dtype="f32")
    assert res["seq_status"][0] == oracle.SEQ_NONFINITE
