"""Which rows a step reads, on the CPU (the oracle's validity rule).

After a rejection the pending proposals are discarded and the next forward
proposes afresh (the schedule under which the closed form of de.news.hada.io,
"Speedup Factor Explorer", holds), so a sequence that rejects reads only its
anchor rows and the rejected token's q row: a NaN in its anchor row N-1 or its
MASK rows changes nothing.  A sequence that keeps every pending token, or had
none, reads rows N-1..2N-2 and fails (every output cleared) if one is unusable.
"""
import numpy as np
import pytest

import oracle


def _rows(seed, N=2, V=8):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((1, 2 * N - 1, V)).astype(np.float32)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_rejecting_sequence_ignores_its_draw_rows(mode):
    N, x = 2, 3
    cur, prev = _rows(1), _rows(2)
    cur[0, 0, x] = -np.inf            # p(x) = 0 and x is not the argmax: rejected in every mode
    bad = cur.copy()
    bad[0, 1, 5] = np.nan             # the bonus row
    bad[0, 2, 0] = np.inf             # the MASK row
    ref = oracle.isd_step(cur, prev, [[x]], [[0.5]], N, 1.0, mode, 3, 4, dtype="f32")
    got = oracle.isd_step(bad, prev, [[x]], [[0.5]], N, 1.0, mode, 3, 4, dtype="f32")
    assert got["seq_status"][0] == oracle.SEQ_OK and got["accepted_len"][0] == 1
    for k in ("accepted_len", "tokens_out", "new_q", "p_out", "accept_margin", "cdf_margin"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("pending", [True, False])
def test_proposing_sequence_fails_on_a_bad_draw_row(mode, pending):
    N = 2
    cur, prev = _rows(5), _rows(6)
    x = int(np.argmax(cur[0, 0]))     # the argmax (kept in greedy mode) ...
    cur[0, 2, 4] = np.nan             # ... and a NaN in the MASK row
    pend, q = ([[x]], [[1e-30]]) if pending else ([[-1]], [[0.0]])  # q tiny: kept when sampled
    got = oracle.isd_step(cur, prev, pend, q, N, 1.0, mode, 3, 4, dtype="f32")
    assert got["seq_status"][0] == oracle.SEQ_NONFINITE
    assert got["accepted_len"][0] == 0 and (got["tokens_out"] == -1).all()
    assert (got["new_q"] == 0).all() and (got["p_out"] == 0).all()
    assert (got["accept_margin"] == -1).all() and (got["cdf_margin"] == -1).all()


def test_bad_anchor_row_fails_a_pending_sequence_only():
    N = 3
    cur, prev = _rows(7, N), _rows(8, N)
    cur = np.concatenate([cur, cur])  # two sequences
    prev = np.concatenate([prev, prev])
    cur[:, 1, 2] = np.nan             # anchor row 1
    got = oracle.isd_step(cur, prev, [[1, 2], [-1, -1]], [[0.5, 0.5], [0.0, 0.0]], N, 1.0, 0, 3, 4, dtype="f32")
    assert got["seq_status"].tolist() == [oracle.SEQ_NONFINITE, oracle.SEQ_OK]
    assert got["accepted_len"].tolist()[1] == 1
