"""Exact enumeration of one ISD forward's outcomes over the 2^-24 uniform lattice.

Test harness.  The oracle is used as a black box: every uniform the step draws
is u = k * 2^-24 with k in [0, 2^24), and each decision is monotone in its own
uniform (an acceptance test u < p/q holds for a prefix of the lattice; an
inverse-CDF index never decreases as u grows).  So the lattice splits into
runs of constant outcome that bisection finds with about 24 oracle calls per
run.  The probability of a run is its length times 2^-24, exactly.
"""
import numpy as np

import oracle

LATTICE = 1 << 24


def runs(decide, lo=0, hi=LATTICE):
    """Split [lo, hi) into maximal runs of constant decide(k) -> [(value, k0, count)].

    decide must be constant on runs that appear in a fixed order (monotone)."""
    out = []
    k = lo
    while k < hi:
        v = decide(k)
        a, b = k, hi - 1  # largest k' in [k, hi) with decide(k') == v
        if decide(b) == v:
            a = b
        else:
            while b - a > 1:
                mid = (a + b) // 2
                if decide(mid) == v:
                    a = mid
                else:
                    b = mid
        out.append((v, k, a - k + 1))
        k = a + 1
    return out


def forward_outcomes(logits, prev_logits, pending, pending_q, N, T, dtype="f32", mode=0):
    """All outcomes of one forward for one sequence, with exact probabilities.

    logits, prev_logits: [2N-1][V]; pending: list of N-1 tokens or None; mode: the
    oracle's greedy argument (0 sampling, 2 argmax proposals with sampled verification).
    Returns [(prob, emitted tokens tuple, new pending tuple or None, new q tuple)].
    """
    R = 2 * N - 1
    lg = np.asarray(logits)[None]
    pv = None if prev_logits is None else np.asarray(prev_logits)[None]
    pt = np.array([pending if pending is not None else [-1] * (N - 1)], dtype=np.int32)
    pq = np.array([pending_q if pending_q is not None else [0.0] * (N - 1)], dtype=np.float32)

    def call(ua, us):
        res = oracle.isd_step_u(lg, pv, pt, pq, N, T, mode, np.array(ua)[None],
                                np.array(us)[None], dtype=dtype)
        assert res["seq_status"][0] == oracle.SEQ_OK
        return res

    outcomes = []

    def proposals(ua, us, j, prob, emitted):
        # MASK row N-1+j, then the next one
        if j == N:
            res = call(ua, us)
            newp = tuple(int(t) for t in res["tokens_out"][0, N:])
            newq = tuple(float(np.float32(x)) for x in res["new_q"][0])
            outcomes.append((prob, emitted, newp, newq))
            return
        r = N - 1 + j

        def dec(k):
            us2 = list(us)
            us2[r] = k / LATTICE
            return int(call(ua, us2)["tokens_out"][0, r])

        for v, k0, cnt in runs(dec):
            us2 = list(us)
            us2[r] = k0 / LATTICE
            proposals(ua, us2, j + 1, prob * cnt / LATTICE, emitted)

    def sample(ua, K, prob):
        # the one inverse-CDF draw of the step: residual row K, or row N-1
        row = K if (pending is not None and K < N - 1) else N - 1
        us = [0.0] * R

        def dec(k):
            us2 = list(us)
            us2[row] = k / LATTICE
            res = call(ua, us2)
            return tuple(int(t) for t in res["tokens_out"][0, :int(res["accepted_len"][0])])

        for emitted, k0, cnt in runs(dec):
            us2 = list(us)
            us2[row] = k0 / LATTICE
            p = prob * cnt / LATTICE
            if pending is not None and K < N - 1:
                outcomes.append((p, emitted, None, None))
            else:
                proposals(ua, us2, 1, p, emitted)

    def accept(i, ua, prob):
        # acceptance test of pending x_i (uniform of row i-1), earlier ones accepted
        if pending is None:
            sample(ua, 0, prob)
            return
        if i == N:
            sample(ua, N - 1, prob)
            return

        def dec(k):
            ua2 = list(ua)
            ua2[i - 1] = k / LATTICE
            return int(call(ua2, [0.0] * R)["accepted_len"][0]) - 1 >= i

        for ok, k0, cnt in runs(dec):
            ua2 = list(ua)
            ua2[i - 1] = k0 / LATTICE
            if ok:
                accept(i + 1, ua2, prob * cnt / LATTICE)
            else:
                sample(ua2, i - 1, prob * cnt / LATTICE)

    accept(1, [0.0] * R, 1.0)
    return outcomes


def softmax(x, T=1.0):
    x = np.asarray(x, dtype=np.float64) / T
    m = np.max(x)
    e = np.exp(x - m)
    return e / e.sum()
