"""GPU parity of the tensor-core LM-head projection and of isd_step_from_hidden
against the fp64 oracle.

Grid inputs (small multiples of 1/8 and 1/256) make every fp32 partial sum
exact, so the kernel must match the oracle bit for bit whatever its summation
order: any operand, layout or index mistake shows.  Gaussian inputs at the full
size (448 query rows, K = 4096, V = 151936) check the rounding: every sampled
logit must be the bf16 rounding of a value within the fp32 accumulation bound
E = K * 2^-22 * sum_k |h_k w_k| of the exact sum, and at least 99% must equal
the oracle's correctly rounded value (accumulation errors are ~1e-3 ulp, so a
boundary is crossed far less often).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import lm_head as olm
from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import grid_hidden_stream, lm_head_inputs
from parity import ParityStats, check_flag_rate, compare_step

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _host(t):
    return olm.bf16_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def _run(h, w):
    hd, wd = _dev(h), _dev(w)
    out = torch.full((h.shape[0], w.shape[0]), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    isd.isd_lm_head(hd, wd, out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return _host(out)


@pytest.mark.parametrize("M,K,V", [
    (32, 128, 256),      # one vocabulary tile pair, two K blocks
    (45, 200, 300),      # ragged everything: K not a multiple of 64, V not of 128, M not of 32
    (7, 64, 1000),
    (448, 4096, 2125),   # the full query-row count and hidden size, ragged vocabulary tail
    (600, 256, 513),     # more than 512 query rows: two blocks
    (300, 128, 31749),   # whole waves of full tiles, then a long tail of tiles with two MMAs each
    (1, 8, 1),           # smallest
])
def test_lm_head_exact_on_grid_inputs(M, K, V):
    h, w = lm_head_inputs(M, K, V, seed=M + K + V, grid=True)
    got = _run(h, w)
    want = olm.lm_head(h, w)
    bad = got != want
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], want[bad][:5])


def _bf16_next(r, up):
    """The bf16 neighbour of bf16 values r (float64) above (up) or below."""
    f = r.astype(np.float32)
    bits = f.view(np.uint32).astype(np.int64) >> 16
    neg = (bits & 0x8000) != 0
    mag = bits & 0x7FFF
    toward_zero = neg == up  # moving up from a negative value, or down from a positive one
    zero = mag == 0
    mag = np.where(toward_zero & ~zero, mag - 1, mag + 1)
    sign = np.where(zero, np.where(up, 0, 0x8000), bits & 0x8000)
    out = ((sign | mag) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return out


def _bf16_below(x):
    """Largest bf16 value <= x (x float64 array)."""
    r = olm.round_bf16(x)
    return np.where(r > x, _bf16_next(r, up=False), r)


def _bf16_above(x):
    """Smallest bf16 value >= x."""
    r = olm.round_bf16(x)
    return np.where(r < x, _bf16_next(r, up=True), r)


def _check_gaussian(got, h, w_rows):
    exact = olm.exact(h, w_rows)
    bound = h.shape[1] * 2.0**-22 * olm.abs_sum(h, w_rows)
    lo, hi = _bf16_below(exact - bound), _bf16_above(exact + bound)
    inside = (got >= lo) & (got <= hi)
    assert inside.all(), (np.argwhere(~inside)[:5], got[~inside][:5], exact[~inside][:5])
    same = np.mean(got == olm.round_bf16(exact))
    assert same >= 0.99, same
    return same


def test_lm_head_gaussian_small():
    h, w = lm_head_inputs(100, 512, 777, seed=11)
    _check_gaussian(_run(h, w), h, w)


def test_lm_head_gaussian_full_size_sampled():
    M, K, V = 448, 4096, 151936
    h, w = lm_head_inputs(M, K, V, seed=2024)
    got_all = torch.empty((M, V), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    isd.isd_lm_head(_dev(h), _dev(w), got_all, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(1)
    # first and last tiles, tile edges, and random rows
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(V - 256, V), np.arange(127, V, 128 * 97),
                                     rng.choice(V, 4096, replace=False)]))
    got = _host(got_all[:, torch.from_numpy(rows).cuda()])
    _check_gaussian(got, h, w[rows])
    assert isd.lm_head_last_launch_count() == 1


@pytest.mark.parametrize("greedy,temperature,B,N,K,V,w_den", [
    (False, 1.0, 6, 4, 256, 1000, 16),      # one partial chunk of 8 tiles, ragged last tile
    (False, 0.7, 6, 4, 256, 1000, 16),
    (True, 1.0, 6, 4, 256, 1000, 16),
    (False, 1.0, 16, 4, 64, 151936, 8),     # 75 chunks, the last of 3 tiles
    (True, 1.0, 16, 4, 64, 151936, 8),
    (False, 1.0, 70, 4, 64, 5000, 8),       # 490 query rows: two projection launches
])
def test_step_from_hidden_matches_oracle_chain(greedy, temperature, B, N, K, V, w_den):
    """Three chained steps: the oracle runs its own projection and its own step.  Grid inputs
    with logits of standard deviation about 3 (w_den), as in the logit workloads."""
    R = 2 * N - 1
    st = isd.StepState(B, N, V, isd.ISD_BF16, from_hidden=True)
    logits = [torch.empty((B, R, V), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    stats = ParityStats()
    prev_ref = None
    _, w = lm_head_inputs(1, K, V, seed=77, grid=True, w_den=w_den)
    wd = _dev(w)
    hs = grid_hidden_stream(B, N, K, 3, seed=100 + B + V)
    for t in range(3):
        h = hs[t].reshape(B * R, K)
        pend, pq = st.pending()
        pend_h, pq_h = pend.cpu().numpy().copy(), pq.cpu().numpy().copy()
        out = st.outputs()
        cur, prev = logits[t % 2], (logits[(t + 1) % 2] if t else None)
        isd.isd_step_from_hidden(_dev(h).view(B, R, K), wd, cur, prev, pend, pq, N, temperature, greedy,
                                 4321, t, *out, p_out=st.p_out, diag=st.diag, workspace=st.workspace)
        st.t += 1
        torch.cuda.synchronize()
        ref_logits = olm.f64_to_bf16_bits(olm.lm_head(h, w)).reshape(B, R, V)
        if not greedy:  # greedy decisions need no whole rows: the logits are not stored then
            np.testing.assert_array_equal(_host(cur).reshape(B, R, V), olm.bf16_to_f64(ref_logits))
        ref = oracle.isd_step(ref_logits, prev_ref, pend_h, pq_h, N, temperature, greedy, 4321, t, dtype="bf16")
        gpu = dict(accepted_len=out[0].cpu().numpy(), tokens_out=out[1].cpu().numpy(),
                   new_q=out[2].cpu().numpy(), p_out=st.p_out.cpu().numpy())
        compare_step(gpu, ref, pend_h, pq_h, N, greedy, temperature, ref_logits, prev_ref, 4321, t, "bf16", stats,
                     where="step %d" % t)
        prev_ref = ref_logits
    assert int(st.diag[isd.DIAG_STATUS].item()) == 0
    check_flag_rate(stats, V)


@pytest.fixture(scope="module")
def full_size_inputs():
    """The from-hidden workload at its full size: B=64, N=4, K=4096, V=151936; hidden states
    N(0, 1) chained across forwards (clean rows = previous MASK rows + N(0, 0.39^2)), weight
    N(0, 0.02^2)."""
    from diffusion_lm_decoding_isd_b300.synthetic import rotating_pool
    B, N, K, V = 64, 4, 4096, 151936
    _, w = lm_head_inputs(1, K, V, seed=31)
    hid = rotating_pool(B, N, K, 1.0, 0.39, 32, 4, "bf16")
    return B, N, K, V, _dev(w), hid


@pytest.fixture(scope="module")
def pool():
    from oracle.parallel import OraclePool
    with OraclePool() as p:
        yield p


def test_step_from_hidden_full_size_on_its_logits(full_size_inputs, pool):
    """Sampling from hidden states at the full size, four chained steps: the oracle's step runs
    on the logits the GPU's projection stored (the step's statistics come from the epilogue, on
    those same bf16 values), every sequence compared with the parity rule of the logits path
    (probabilities within 1e-5).  The projection's own accuracy is checked against the exact
    sums by test_lm_head_gaussian_full_size_sampled; here the logits the standalone projection
    writes are also required to be bit-identical to those the fused step stored."""
    B, N, K, V, wd, hid = full_size_inputs
    R = 2 * N - 1
    st = isd.StepState(B, N, V, isd.ISD_BF16, from_hidden=True)
    logits = [torch.empty((B, R, V), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    stats = ParityStats()
    prev_h = None
    for t in range(4):
        pend, pq = st.pending()
        pend_h, pq_h = pend.cpu().numpy().copy(), pq.cpu().numpy().copy()
        out = st.outputs()
        hd = _dev(hid[t]).view(B, R, K)
        isd.isd_step_from_hidden(hd, wd, logits[t & 1], logits[(t - 1) & 1] if t else None, pend, pq,
                                 N, 1.0, False, 99, t, *out, p_out=st.p_out, diag=st.diag, workspace=st.workspace)
        st.t += 1
        torch.cuda.synchronize()
        host = logits[t & 1].view(torch.int16).cpu().numpy().view(np.uint16)
        if t == 0:
            alone = torch.empty((B * R, V), dtype=torch.bfloat16, device="cuda")
            isd.isd_lm_head(hd.view(B * R, K), wd, alone)
            torch.cuda.synchronize()
            assert torch.equal(alone.view(torch.int16).view(B, R, V), logits[0].view(torch.int16))
        gpu = dict(accepted_len=out[0].cpu().numpy(), tokens_out=out[1].cpu().numpy(),
                   new_q=out[2].cpu().numpy(), p_out=st.p_out.cpu().numpy())
        ref = pool.isd_step(host, prev_h, pend_h, pq_h, N, 1.0, False, 99, t, dtype="bf16")
        assert (ref["seq_status"] == 0).all()
        compare_step(gpu, ref, pend_h, pq_h, N, False, 1.0, host, prev_h, 99, t, "bf16", stats, where="step %d" % t)
        prev_h = host
    assert int(st.diag[isd.DIAG_STATUS].item()) == 0
    check_flag_rate(stats, V)
    assert stats.tests > 0


def test_step_from_hidden_full_size_greedy(full_size_inputs, pool):
    """Greedy decoding from hidden states at the full size (K = 4096), four chained steps.  The
    step stores no logits in this mode, so the oracle's step runs on the standalone
    projection's logits of the same hidden states (bit-identical to those the fused
    projection computes, checked in the sampling test); argmax decisions must agree exactly."""
    B, N, K, V, wd, hid = full_size_inputs
    R = 2 * N - 1
    st = isd.StepState(B, N, V, isd.ISD_BF16, from_hidden=True)
    logits = [torch.empty((B, R, V), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    alone = torch.empty((B * R, V), dtype=torch.bfloat16, device="cuda")
    stats = ParityStats()
    for t in range(4):
        pend, pq = st.pending()
        pend_h, pq_h = pend.cpu().numpy().copy(), pq.cpu().numpy().copy()
        out = st.outputs()
        hd = _dev(hid[t]).view(B, R, K)
        isd.isd_step_from_hidden(hd, wd, logits[t & 1], logits[(t - 1) & 1] if t else None, pend, pq,
                                 N, 1.0, True, 99, t, *out, p_out=st.p_out, diag=st.diag, workspace=st.workspace)
        st.t += 1
        isd.isd_lm_head(hd.view(B * R, K), wd, alone)
        torch.cuda.synchronize()
        host = alone.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, R, V)
        gpu = dict(accepted_len=out[0].cpu().numpy(), tokens_out=out[1].cpu().numpy(),
                   new_q=out[2].cpu().numpy(), p_out=st.p_out.cpu().numpy())
        ref = pool.isd_step(host, None, pend_h, pq_h, N, 1.0, True, 99, t, dtype="bf16")
        compare_step(gpu, ref, pend_h, pq_h, N, True, 1.0, host, None, 99, t, "bf16", stats, where="step %d" % t)
    assert int(st.diag[isd.DIAG_STATUS].item()) == 0
    assert stats.tests > 0 and stats.accepts > 0
