"""GPU-vs-oracle parity harness (test infrastructure).

Each step runs the CUDA path and then the fp64 oracle on identical bytes and the
identical pending state the GPU carried (teacher forcing, so one divergence
cannot cascade).  Every output of every sequence is compared:

- Decisions the oracle does not flag as near-ties must agree exactly.
- An inverse-CDF draw whose target lies within 1e-6 (relative to the sum of
  the weights) of a CDF edge is flagged; the GPU token must then lie in the
  range of tokens whose CDF interval comes within that window of the target
  (the oracle returns the range), and the new q of a proposal drawn there must
  be the oracle's probability of the token the GPU drew.
- An acceptance test with |u - p/q| < 1e-6 is flagged; if the GPU decided it the
  other way, the oracle is run again on that sequence with the uniform of that
  test moved across p/q, and the GPU must match that run exactly (with the same
  near-tie rules for its draws).
- Probabilities (new q, p of pending tokens) must agree to 1e-5 relative.

Counts of decisions, flags and GPU/oracle differences are kept for the flag-rate
rule (see check_flag_rate).
"""
import itertools

import numpy as np
import torch

import oracle
from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream

PROB_RTOL = 1e-5
NEAR = oracle.NEAR_TOL


def to_device(host, dtype):
    if dtype == "bf16":
        return torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(host)).cuda()


class ParityStats:
    def __init__(self):
        self.acc_decisions = 0    # acceptance tests made
        self.acc_flagged = 0      # ... within NEAR of u = p/q
        self.acc_flipped = 0      # ... decided the other way by the GPU (all flagged)
        self.cdf_decisions = 0    # inverse-CDF draws made
        self.cdf_flagged = 0      # ... whose target is within NEAR of a CDF edge
        self.cdf_differ = 0       # ... where the GPU drew another token (all flagged)
        self.max_differ_margin = 0.0  # largest oracle margin of a draw the GPU took differently
        self.seq_steps = 0
        self.emitted = 0
        self.accepts = 0
        self.tests = 0

    @property
    def decisions(self):
        return self.acc_decisions + self.cdf_decisions

    def __repr__(self):
        return ("acceptance tests %d (flagged %d, decided otherwise %d); draws %d (flagged %d = %.2e, "
                "drawn otherwise %d = %.2e, largest margin of those %.2e); seq_steps=%d emitted=%d "
                "accept_rate=%.4f"
                % (self.acc_decisions, self.acc_flagged, self.acc_flipped, self.cdf_decisions,
                   self.cdf_flagged, self.cdf_flagged / max(1, self.cdf_decisions), self.cdf_differ,
                   self.cdf_differ / max(1, self.cdf_decisions), self.max_differ_margin, self.seq_steps,
                   self.emitted, self.accepts / max(1, self.tests)))


def check_flag_rate(stats, V):
    """The flag-rate rule.

    Acceptance tests: the benchmark spec's rule as written.  A test is within 1e-6 of
    u = p/q with probability about 2e-6, so flagged tests stay below 1e-4 of
    the tests.

    Inverse-CDF draws: the share of draws flagged by a 1e-6 window (relative to
    the sum of the weights) is a property of the input, not of the kernel: every
    token lighter than 2e-6 of the mass lies entirely inside the window, so a
    draw landing on one is always flagged.  Over V = 151936 tokens most tokens
    are that light (the mean is 6.6e-6), and the measured share is 1.5% (T=0.7)
    to 7% (T=1) of draws on the synthetic rows; 1e-4 of decisions is out of
    reach for any implementation, the fp64 oracle included, so it is not
    asserted.  What is asserted instead: every flagged draw is checked for
    validity (the GPU token lies in the window's token range), every unflagged
    draw matches exactly, and the draws the GPU took differently are few: with
    the GPU's CDF edges within delta * sum(w) of the oracle's (measured delta
    below 1e-8), a draw can differ only when its target lies within delta of
    one of the V edges, so at most V * delta of the draws; the bound asserted
    is V * 1e-8, and at least 2 draws.
    """
    assert stats.acc_flagged <= max(1, 1e-4 * stats.acc_decisions), stats
    assert stats.cdf_differ <= max(2, V * 1e-8 * stats.cdf_decisions), stats
    print(stats)


def _draw_position(r, N, has_pending):
    """Position in tokens_out of the token drawn at row r."""
    return 0 if (r == N - 1 and not has_pending) else r


def _compare_sequence(b, gpu, ref, rb, pend_h, N, greedy, T, host, dtype, stats, ctx, prob_rtol):
    """Compare sequence b of the GPU outputs with row rb of the oracle result `ref`."""
    acc_g, tok_g, nq_g = gpu["accepted_len"][b], gpu["tokens_out"][b], gpu["new_q"][b]
    R = 2 * N - 1
    has_pending = pend_h[b, 0] >= 0
    assert acc_g == ref["accepted_len"][rb], (ctx, acc_g, ref["accepted_len"][rb], tok_g, ref["tokens_out"][rb])
    cm, lo, hi = ref["cdf_margin"][rb], ref["cdf_lo"][rb], ref["cdf_hi"][rb]
    drawn = {}  # position -> row of each draw
    for r in range(R):
        if cm[r] >= 0:
            drawn[_draw_position(r, N, has_pending)] = r
    for pos in range(R):
        want = ref["tokens_out"][rb, pos]
        r = drawn.get(pos)
        if r is not None and cm[r] < NEAR:
            assert lo[r] <= tok_g[pos] <= hi[r], (ctx, "flagged draw out of its window", pos, tok_g[pos],
                                                  want, lo[r], hi[r], cm[r])
            if tok_g[pos] != want:
                stats.cdf_differ += 1
                stats.max_differ_margin = max(stats.max_differ_margin, float(cm[r]))
        else:
            assert tok_g[pos] == want, (ctx, pos, tok_g, ref["tokens_out"][rb])
    for j in range(1, N):
        pos = N - 1 + j
        want = ref["new_q"][rb, j - 1]
        if tok_g[pos] >= 0 and tok_g[pos] != ref["tokens_out"][rb, pos]:
            # a flagged proposal drawn at a neighbouring token: its q is that token's p
            want = oracle.softmax_prob(host[b, pos], T, int(tok_g[pos]), dtype)
        np.testing.assert_allclose(nq_g[j - 1], want, rtol=prob_rtol, atol=0, err_msg=ctx)


def _flipped_variants(b, ref, host, prev_h, pend_h, pq_h, N, T, greedy, seed, step, dtype):
    """Oracle runs of sequence b with each nonempty subset of its flagged acceptance tests
    decided the other way (the test's uniform moved to 0, always kept, or 2, never kept)."""
    R = 2 * N - 1
    am = ref["accept_margin"][b]
    flagged = [i for i in range(N - 1) if 0 <= am[i] < NEAR]
    K = int(ref["accepted_len"][b]) - 1  # tests 0..K-1 were kept, test K (if made) rejected
    ua = np.zeros((1, R))
    us = np.zeros((1, R))
    for r in range(R):
        ua[0, r], us[0, r] = oracle.row_uniforms(seed, step, b, r)
    out = []
    for n in range(1, len(flagged) + 1):
        for sub in itertools.combinations(flagged, n):
            u = ua.copy()
            for i in sub:
                u[0, i] = 2.0 if i < K else 0.0
            out.append(oracle.isd_step_u(host[b:b + 1], None if prev_h is None else prev_h[b:b + 1],
                                         pend_h[b:b + 1], pq_h[b:b + 1], N, T, greedy, u, us, dtype=dtype))
    return out


def compare_step(gpu, ref, pend_h, pq_h, N, greedy, T, host, prev_h, seed, step, dtype, stats, where="",
                 prob_rtol=PROB_RTOL):
    """Compare one step's GPU outputs (numpy dict) with the oracle's, every sequence."""
    am, cm = ref["accept_margin"], ref["cdf_margin"]
    stats.acc_decisions += int((am >= 0).sum())
    stats.acc_flagged += int(((am >= 0) & (am < NEAR)).sum())
    stats.cdf_decisions += int((cm >= 0).sum())
    stats.cdf_flagged += int(((cm >= 0) & (cm < NEAR)).sum())
    B = gpu["accepted_len"].shape[0]
    for b in range(B):
        stats.seq_steps += 1
        ctx = "%s seq %d" % (where, b)
        if int(greedy) != isd.ISD_GREEDY:  # sampled verification: the anchor probabilities are reported
            np.testing.assert_allclose(gpu["p_out"][b], ref["p_out"][b], rtol=prob_rtol, atol=1e-30, err_msg=ctx)
        if gpu["accepted_len"][b] == ref["accepted_len"][b]:
            _compare_sequence(b, gpu, ref, b, pend_h, N, greedy, T, host, dtype, stats, ctx, prob_rtol)
        else:
            # only a flagged acceptance test decided the other way may explain it
            variants = [v for v in _flipped_variants(b, ref, host, prev_h, pend_h, pq_h, N, T, greedy, seed, step,
                                                     dtype)
                        if v["accepted_len"][0] == gpu["accepted_len"][b]]
            assert variants, (ctx, "accepted_len differs and no flagged test explains it",
                              gpu["accepted_len"][b], ref["accepted_len"][b], ref["accept_margin"][b])
            stats.acc_flipped += 1
            _compare_sequence(b, gpu, variants[0], 0, pend_h, N, greedy, T, host, dtype, stats, ctx + " (flipped)",
                              prob_rtol)
        acc = int(gpu["accepted_len"][b])
        stats.emitted += acc
        if pend_h[b, 0] >= 0 and ref["seq_status"][b] == 0:
            stats.accepts += acc - 1
            stats.tests += min(acc, N - 1)


def run_parity(B, N, V, dtype="bf16", sigma_l=3.0, sigma_n=0.5, temperature=1.0, greedy=False,
               steps=8, seed=0, philox_seed=1234, stream_gen=None, stats=None, step_of=None, pool=None,
               fused=False):
    """Run `steps` teacher-forced steps and compare every one with the oracle.
    step_of(t) gives the Philox step number of the t-th call (default t); `pool`
    (an oracle.parallel.OraclePool) runs the oracle over the host cores; fused runs
    isd_step_fused instead of isd_step."""
    step_of = step_of or (lambda t: t)
    stats = stats or ParityStats()
    gen = stream_gen or ForwardStream(B, N, V, sigma_l, sigma_n, seed, dtype)
    code = isd.ISD_BF16 if dtype == "bf16" else isd.ISD_F32
    state = isd.StepState(B, N, V, code, fused=fused)
    prev_h = prev_d = None
    ref_step = pool.isd_step if pool is not None else oracle.isd_step
    for t in range(steps):
        host = gen.next()
        dev = to_device(host, dtype)
        pend, pq = state.pending()
        pend_h = pend.cpu().numpy().copy()
        pq_h = pq.cpu().numpy().copy()
        # argmax proposals never read the previous forward: pass none, as a caller may
        no_prev = int(greedy) == isd.ISD_ARGMAX_PROPOSE
        acc, tok, nq = state.step(dev, None if no_prev else prev_d, temperature, greedy, philox_seed,
                                  step=step_of(t))
        torch.cuda.synchronize()
        gpu = dict(accepted_len=acc.cpu().numpy(), tokens_out=tok.cpu().numpy(),
                   new_q=nq.cpu().numpy(), p_out=state.p_out.cpu().numpy())
        pv = None if no_prev else prev_h
        ref = ref_step(host, pv, pend_h, pq_h, N, temperature, greedy, philox_seed, step_of(t), dtype=dtype)
        assert (ref["seq_status"] == 0).all()
        compare_step(gpu, ref, pend_h, pq_h, N, greedy, temperature, host, pv, philox_seed, step_of(t), dtype,
                     stats, where="step %d" % t)
        prev_h, prev_d = host, dev
    diag = state.diag.cpu().numpy()
    assert diag[isd.DIAG_STATUS] == 0, diag
    return stats, diag
