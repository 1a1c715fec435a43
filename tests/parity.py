"""GPU-vs-oracle parity harness (test infrastructure).

Each step runs the CUDA path and then the fp64 oracle on identical bytes and the
identical pending state the GPU carried (teacher forcing, so one divergence
cannot cascade).  Decisions must agree exactly unless the oracle flags them as
near-ties (|u - p/q| or a CDF margin below 1e-6); flagged sequences are counted
and excluded.  Probabilities (new q, p of pending tokens) must agree to 1e-5
relative.
"""
import numpy as np
import torch

import oracle
from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream

PROB_RTOL = 1e-5


def to_device(host, dtype):
    if dtype == "bf16":
        return torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(host)).cuda()


class ParityStats:
    def __init__(self):
        self.decisions = 0
        self.flagged = 0
        self.acc_decisions = 0
        self.cdf_decisions = 0
        self.acc_flagged = 0
        self.cdf_flagged = 0
        self.seq_steps = 0
        self.emitted = 0
        self.accepts = 0
        self.tests = 0

    def __repr__(self):
        return ("decisions=%d (acc %d, cdf %d) flagged seqs=%d (acc %d, cdf %d) seq_steps=%d "
                "emitted=%d accept_rate=%.4f"
                % (self.decisions, self.acc_decisions, self.cdf_decisions, self.flagged,
                   self.acc_flagged, self.cdf_flagged, self.seq_steps, self.emitted,
                   self.accepts / max(1, self.tests)))


def compare_step(gpu, ref, pend_h, N, greedy, stats, where="", prob_rtol=PROB_RTOL):
    """Compare one step's GPU outputs (numpy dict) with the oracle's."""
    acc_g, tok_g, nq_g, pout_g = gpu["accepted_len"], gpu["tokens_out"], gpu["new_q"], gpu["p_out"]
    flags = oracle.near_tie_flags(ref)
    stats.decisions += oracle.decision_count(ref)
    stats.flagged += int(flags.sum())
    na, nc = oracle.decision_counts(ref)
    fa, fc = oracle.near_tie_counts(ref)
    stats.acc_decisions += na
    stats.cdf_decisions += nc
    stats.acc_flagged += fa
    stats.cdf_flagged += fc
    B = acc_g.shape[0]
    for b in range(B):
        stats.seq_steps += 1
        if flags[b]:
            continue
        ctx = "%s seq %d" % (where, b)
        assert acc_g[b] == ref["accepted_len"][b], (ctx, acc_g[b], ref["accepted_len"][b],
                                                     tok_g[b], ref["tokens_out"][b])
        assert (tok_g[b] == ref["tokens_out"][b]).all(), (ctx, tok_g[b], ref["tokens_out"][b])
        np.testing.assert_allclose(nq_g[b], ref["new_q"][b], rtol=prob_rtol, atol=0, err_msg=ctx)
        if int(greedy) != 1:  # sampled verification: the anchor probabilities are reported
            np.testing.assert_allclose(pout_g[b], ref["p_out"][b], rtol=prob_rtol, atol=1e-30,
                                       err_msg=ctx)
        stats.emitted += int(acc_g[b])
        if pend_h[b, 0] >= 0 and ref["seq_status"][b] == 0:
            k = int(acc_g[b]) - 1
            stats.accepts += k
            stats.tests += min(k + 1, N - 1)


def run_parity(B, N, V, dtype="bf16", sigma_l=3.0, sigma_n=0.5, temperature=1.0, greedy=False,
               steps=8, seed=0, philox_seed=1234, stream_gen=None, stats=None, step_of=None):
    """Run `steps` teacher-forced steps and compare every one with the oracle.
    step_of(t) gives the Philox step number of the t-th call (default t)."""
    step_of = step_of or (lambda t: t)
    stats = stats or ParityStats()
    gen = stream_gen or ForwardStream(B, N, V, sigma_l, sigma_n, seed, dtype)
    code = isd.ISD_BF16 if dtype == "bf16" else isd.ISD_F32
    state = isd.StepState(B, N, V, code)
    prev_h = prev_d = None
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
        ref = oracle.isd_step(host, None if no_prev else prev_h, pend_h, pq_h, N, temperature, greedy, philox_seed,
                              step_of(t), dtype=dtype)
        assert (ref["seq_status"] == 0).all()
        compare_step(gpu, ref, pend_h, N, greedy, stats, where="step %d" % t)
        prev_h, prev_d = host, dev
    diag = state.diag.cpu().numpy()
    assert diag[isd.DIAG_STATUS] == 0, diag
    return stats, diag
