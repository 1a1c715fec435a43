"""Monte-Carlo tokens-per-forward of the oracle against the pages' closed form.

de.news.hada.io, "Speedup Factor Explorer": in the memory-bound regime the
speedup is about TPF = (2 + p + ... + p^(N-2)) / (2 - p^(N-1)); the same page
("Durchsatz") and the ai.arkapp.pw blog (compute-efficiency paragraph) print
TPF ~ 2.9 and efficiency TPF^2/(2N-1) ~ 1.22 for N=4, p=0.9.

Rows are built so that every pending token is accepted with probability
exactly alpha: q uniform on tokens 0..m-1, p = alpha*q + (1-alpha)*delta_m,
so sum_x min(p, q) = alpha.
"""
import numpy as np
import pytest

import oracle


def closed_form_tpf(N, p):
    num = 2.0 + sum(p ** k for k in range(1, N - 1))
    return num / (2.0 - p ** (N - 1))


def _rows(N, alpha, m):
    V = m + 1
    R = 2 * N - 1
    q = np.zeros(V)
    q[:m] = 1.0 / m
    p = alpha * q
    p[m] += 1.0 - alpha
    with np.errstate(divide="ignore"):
        lp = np.log(p).astype(np.float32)
        lq = np.log(q).astype(np.float32)
    rows = np.empty((R, V), dtype=np.float32)
    rows[:N] = lp  # verify rows and the anchor row
    rows[N:] = lq  # MASK rows
    return rows


def simulate_tpf(N, alpha, B=2000, steps=120, burn=20, m=8, seed=1234):
    R = 2 * N - 1
    rows = _rows(N, alpha, m)
    logits = np.ascontiguousarray(np.broadcast_to(rows, (B, R, rows.shape[1])))
    pending = -np.ones((B, N - 1), dtype=np.int32)
    pq = np.zeros((B, N - 1), dtype=np.float32)
    per_seq = np.zeros(B)
    for t in range(steps):
        res = oracle.isd_step(logits, logits, pending, pq, N, 1.0, False, seed, t, dtype="f32")
        assert (res["seq_status"] == 0).all()
        if t >= burn:
            per_seq += res["accepted_len"]
        pending = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)
    per_seq /= (steps - burn)
    return per_seq.mean(), per_seq.std(ddof=1) / np.sqrt(B)


@pytest.mark.parametrize("N", [2, 3, 4, 8])
@pytest.mark.parametrize("alpha", [0.5, 0.9, 0.99])
def test_tpf_matches_closed_form(N, alpha):
    tpf, se = simulate_tpf(N, alpha)
    expect = closed_form_tpf(N, alpha)
    assert abs(tpf - expect) < 4.0 * se + 1e-9, (tpf, expect, se)


def test_printed_values_n4_p09():
    # the pages print TPF ~ 2.9 and efficiency ~ 1.22 at N=4, p=0.9
    tpf = closed_form_tpf(4, 0.9)
    assert abs(tpf - 2.9) < 0.05
    assert abs(tpf ** 2 / 7 - 1.22) < 0.01
    sim, se = simulate_tpf(4, 0.9, B=4000, steps=150)
    assert abs(sim - 2.9) < 0.05
    assert abs(sim ** 2 / 7 - 1.22) < 0.02


def test_closed_form_edges():
    # N=2: the p-sum is empty, TPF = 2/(2-p); p=1 gives N tokens per forward
    assert closed_form_tpf(2, 0.5) == pytest.approx(2 / 1.5)
    for N in (2, 3, 4, 8):
        assert closed_form_tpf(N, 1.0) == pytest.approx(N)
        assert closed_form_tpf(N, 0.0) == pytest.approx(1.0)



def _rows_argmax(N, alpha, m):
    """Argmax proposals (mode 2) accepted with probability exactly alpha: the MASK rows'
    argmax is token 0, and every anchor row gives token 0 probability alpha."""
    V = m + 1
    R = 2 * N - 1
    p = np.full(V, (1.0 - alpha) / m)
    p[0] = alpha
    q = np.zeros(V)
    q[0] = 1.0
    rows = np.empty((R, V), dtype=np.float32)
    rows[:N] = np.log(p).astype(np.float32)
    rows[N:] = q.astype(np.float32)
    return rows


@pytest.mark.parametrize("N", [2, 4, 8])
@pytest.mark.parametrize("alpha", [0.5, 0.9])
def test_argmax_proposals_tpf_matches_closed_form(N, alpha):
    R = 2 * N - 1
    B, steps, burn = 2000, 120, 20
    rows = _rows_argmax(N, alpha, 8)
    logits = np.ascontiguousarray(np.broadcast_to(rows, (B, R, rows.shape[1])))
    pending = -np.ones((B, N - 1), dtype=np.int32)
    pq = np.zeros((B, N - 1), dtype=np.float32)
    per_seq = np.zeros(B)
    for t in range(steps):
        res = oracle.isd_step(logits, None, pending, pq, N, 1.0, 2, 99, t, dtype="f32")
        assert (res["seq_status"] == 0).all()
        if t >= burn:
            per_seq += res["accepted_len"]
        pending = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)
        assert (pending[pending >= 0] == 0).all() and (pq[pending >= 0] == 1.0).all()
    per_seq /= (steps - burn)
    se = per_seq.std(ddof=1) / np.sqrt(B)
    assert abs(per_seq.mean() - closed_form_tpf(N, alpha)) < 4.0 * se + 1e-9


def test_argmax_proposals_replacement_is_never_the_rejected_token():
    N, V = 2, 8
    rows = _rows_argmax(N, 0.5, V - 1)
    B = 500
    logits = np.ascontiguousarray(np.broadcast_to(rows, (B, 3, V)))
    pending = np.zeros((B, 1), dtype=np.int32)  # token 0 pending, q = 1
    pq = np.ones((B, 1), dtype=np.float32)
    res = oracle.isd_step(logits, None, pending, pq, N, 1.0, 2, 5, 0, dtype="f32")
    rejected = res["accepted_len"] == 1
    assert rejected.any() and (~rejected).any()
    assert (res["tokens_out"][rejected, 0] != 0).all()
    assert (res["tokens_out"][~rejected, 0] == 0).all()
