"""CUDA path vs the fp64 oracle, element by element, on seeded synthetic inputs."""
import numpy as np
import pytest
import torch

import oracle
from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream, f32_to_bf16_bits
from oracle.parallel import OraclePool
from parity import check_flag_rate, run_parity, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    """The oracle over the host cores (spawned worker processes)."""
    with OraclePool() as p:
        yield p


def test_tiny_fp32_config():
    # B=1, N=2, V=256, fp32 logits N(0, 2^2), anchors = proposals + N(0, 0.3^2), T=1, 64 steps
    stats, diag = run_parity(1, 2, 256, "f32", 2.0, 0.3, 1.0, False, steps=64, seed=0)
    check_flag_rate(stats, 256)
    assert stats.tests > 20


def test_b8_n4_full_vocab(pool):
    # B=8, N=4, V=151936 bf16 N(0, 3^2), anchors + N(0, 0.5^2), T=1, all 256 steps
    stats, diag = run_parity(8, 4, 151936, "bf16", 3.0, 0.5, 1.0, False, steps=256, seed=1, pool=pool)
    check_flag_rate(stats, 151936)
    assert 0.6 < stats.accepts / stats.tests < 0.95


@pytest.mark.parametrize("greedy,temperature", [(True, 1.0), (False, 0.7), (isd.ISD_ARGMAX_PROPOSE, 1.0)])
def test_b64_n4_full_vocab(greedy, temperature, pool):
    # B=64, N=4, V=151936 bf16, 64 consecutive steps of each mode
    stats, diag = run_parity(64, 4, 151936, "bf16", 3.0, 0.5, temperature, greedy, steps=64, seed=2, pool=pool)
    check_flag_rate(stats, 151936)


def test_b8_n4_full_vocab_argmax_proposals():
    """Argmax proposals verified by sampling: every rejection draws from the anchor row
    without the rejected token (no previous row is passed)."""
    stats, diag = run_parity(8, 4, 151936, "bf16", 3.0, 0.5, 1.0, isd.ISD_ARGMAX_PROPOSE, steps=30, seed=6)
    check_flag_rate(stats, 151936)
    assert diag[isd.DIAG_RESIDUALS] > 0 and stats.accepts > 0


def test_q_row_statistics_reread_when_not_chained():
    """The workspace keeps the MASK rows' statistics for the next call only when that call
    names this call's logits as prev_logits with step + 1.  With step numbers that skip,
    every residual re-reads its q row: the results must still match the oracle."""
    stats, diag = run_parity(8, 4, 151936, "bf16", 3.0, 0.5, 1.0, False, steps=12, seed=4,
                             step_of=lambda t: 3 * t + 1)
    check_flag_rate(stats, 151936)
    assert diag[isd.DIAG_RESIDUALS] > 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_residual_with_more_chunks_than_shared_memory_holds(dtype, pool):
    """A vocabulary of 1.1 M entries: 538 (bf16) or 1075 (fp32) chunks per row, more than the
    decision pass keeps in shared memory for a residual (512), so the residual's chunk sums go
    through global memory with an atomic total; the outputs must still match the oracle."""
    stats, diag = run_parity(8, 2, 1_100_000, dtype, 3.0, 1.0, 1.0, False, steps=6, seed=9, pool=pool)
    check_flag_rate(stats, 1_100_000)
    assert diag[isd.DIAG_RESIDUALS] > 0


SMALL = [
    # B, N, V, dtype, sigma_n, T
    (5, 2, 2048 * 3 + 136, "bf16", 0.5, 1.0),   # several chunks and a ragged tail
    (3, 3, 1000, "bf16", 0.1, 0.5),             # one partial chunk, high acceptance
    (4, 4, 1001, "bf16", 2.0, 1.0),             # V*2 not a multiple of 16: scalar loads
    (2, 8, 5000, "f32", 0.5, 2.0),              # fp32, N=8 (15 rows)
    (3, 4, 1023, "f32", 0.5, 1.0),              # fp32 unaligned rows
    (37, 3, 4096, "bf16", 1.0, 1.0),            # exact chunk multiple
    (2, 32, 300, "bf16", 0.5, 1.0),             # the largest stride
    (1, 2, 7, "bf16", 0.5, 1.0),                # V smaller than a vector
    (2, 3, 1, "f32", 0.5, 1.0),                 # a single-token vocabulary
]


@pytest.mark.parametrize("B,N,V,dtype,sigma_n,T", SMALL)
@pytest.mark.parametrize("greedy", [isd.ISD_SAMPLE, isd.ISD_GREEDY, isd.ISD_ARGMAX_PROPOSE])
def test_small_shapes(B, N, V, dtype, sigma_n, T, greedy):
    stats, diag = run_parity(B, N, V, dtype, 2.0, sigma_n, T, greedy, steps=12, seed=B * 7 + N)
    check_flag_rate(stats, V)


def test_many_sequences_small_vocab():
    stats, diag = run_parity(3000, 4, 64, "bf16", 2.0, 0.5, 1.0, False, steps=4, seed=5)
    check_flag_rate(stats, 64)


def test_masked_vocab_rows():
    """Rows where most of the vocabulary is -inf (one or a few allowed tokens)."""
    B, N, V = 6, 3, 3000
    R = 2 * N - 1
    rng = np.random.default_rng(17)

    class Masked:
        def __init__(self):
            self.inner = ForwardStream(B, N, V, 2.0, 0.5, 3, "f32")

        def next(self):
            x = self.inner.next().copy()
            for b in range(B):
                for r in range(R):
                    keep = rng.choice(V, size=1 + (b % 3) * 5, replace=False)
                    row = np.full(V, -np.inf, dtype=np.float32)
                    row[keep] = x[b, r, keep]
                    x[b, r] = row
            return x

    stats, diag = run_parity(B, N, V, "f32", steps=10, stream_gen=Masked())
    check_flag_rate(stats, V)
    rng = np.random.default_rng(17)
    stats, diag = run_parity(B, N, V, "f32", steps=10, stream_gen=Masked(), greedy=isd.ISD_ARGMAX_PROPOSE)
    check_flag_rate(stats, V)


def test_deterministic_across_runs():
    outs = []
    for _ in range(2):
        gen = ForwardStream(16, 4, 20000, 3.0, 0.5, 9, "bf16")
        st = isd.StepState(16, 4, 20000)
        prev = None
        rec = []
        for t in range(6):
            dev = to_device(gen.next(), "bf16")
            acc, tok, nq = st.step(dev, prev, 1.0, False, 99)
            rec.append((acc.cpu().numpy().copy(), tok.cpu().numpy().copy(), nq.cpu().numpy().copy()))
            prev = dev
        outs.append(rec)
    for a, b in zip(*outs):
        for x, y in zip(a, b):
            assert (x == y).all()


def _one_step(host, prev_host, pend, pq, N, T, greedy, dtype="f32"):
    B, R, V = host.shape
    dev = to_device(host, dtype)
    prev = None if prev_host is None else to_device(prev_host, dtype)
    st = isd.StepState(B, N, V, isd.ISD_F32 if dtype == "f32" else isd.ISD_BF16)
    st.start_pending.copy_(torch.from_numpy(np.asarray(pend, dtype=np.int32)))
    st.start_q.copy_(torch.from_numpy(np.asarray(pq, dtype=np.float32)))
    acc, tok, nq = st.step(dev, prev, T, greedy, 5)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), tok.cpu().numpy(), nq.cpu().numpy(), st.diag.cpu().numpy()


def test_nonfinite_and_bad_pending():
    N, V, B = 2, 512, 4
    rng = np.random.default_rng(0)
    host = rng.standard_normal((B, 3, V)).astype(np.float32)
    prev = rng.standard_normal((B, 3, V)).astype(np.float32)
    host[1, 0, 100] = np.nan     # seq 1 has pending tokens: row 0 is read -> error
    host[2, 0, 7] = np.inf       # seq 2 has none: row 0 is not read -> fine
    host[3, 2, 9] = np.inf       # a MASK row is always read -> error
    pend = [[3], [3], [-1], [-1]]
    pq = [[0.01], [0.01], [0.0], [0.0]]
    for greedy in (False, True):
        acc, tok, nq, diag = _one_step(host, prev, pend, pq, N, 1.0, greedy)
        assert acc[1] == 0 and (tok[1] == -1).all()
        assert acc[3] == 0 and (tok[3] == -1).all()
        assert acc[0] >= 1 and acc[2] == 1
        assert diag[isd.DIAG_STATUS] == isd.ISD_ERR_NONFINITE
        ref = oracle.isd_step(host, prev, pend, pq, N, 1.0, greedy, 5, 0, dtype="f32")
        assert ref["seq_status"].tolist() == [0, 1, 0, 1]
        assert acc.tolist() == ref["accepted_len"].tolist()
        assert (tok == ref["tokens_out"]).all()
    # a pending token out of range, and a non-positive q
    acc, tok, nq, diag = _one_step(host[:1], prev[:1], [[V]], [[0.5]], N, 1.0, False)
    assert acc[0] == 0 and diag[isd.DIAG_STATUS] == isd.ISD_ERR_BAD_PENDING
    acc, tok, nq, diag = _one_step(host[:1], prev[:1], [[2]], [[0.0]], N, 1.0, False)
    assert acc[0] == 0 and diag[isd.DIAG_STATUS] == isd.ISD_ERR_BAD_PENDING


def test_residual_q_row_nonfinite():
    """A rejected token whose q row (previous MASK row N+K) holds NaN fails the sequence."""
    N, V = 2, 256
    host = np.zeros((1, 3, V), dtype=np.float32)
    host[0, 0, :] = -np.inf
    host[0, 0, 0] = 0.0           # p is a point mass on token 0
    prev = np.zeros((1, 3, V), dtype=np.float32)
    prev[0, 2, 5] = np.nan        # the q row
    acc, tok, nq, diag = _one_step(host, prev, [[4]], [[0.5]], N, 1.0, False)
    ref = oracle.isd_step(host, prev, [[4]], [[0.5]], N, 1.0, False, 5, 0, dtype="f32")
    assert ref["seq_status"][0] == oracle.SEQ_NONFINITE
    assert acc[0] == 0 and (tok[0] == -1).all()
    assert diag[isd.DIAG_STATUS] == isd.ISD_ERR_NONFINITE


def test_greedy_stream_is_stepwise_argmax():
    """Greedy mode: every emitted token is the argmax of the anchor row of its position."""
    B, N, V = 16, 4, 151936
    gen = ForwardStream(B, N, V, 3.0, 0.25, 21, "bf16")
    st = isd.StepState(B, N, V)
    prev = None
    for t in range(8):
        host = gen.next()
        dev = to_device(host, "bf16")
        pend, _ = st.pending()
        pend_h = pend.cpu().numpy().copy()
        acc, tok, nq = st.step(dev, prev, 1.0, True, 0)
        acc, tok = acc.cpu().numpy(), tok.cpu().numpy()
        amax = host.view(np.int16)  # argmax over bf16 values via float
        vals = (host.astype(np.uint32) << 16).view(np.float32)
        am = vals.argmax(axis=2)
        for b in range(B):
            if pend_h[b, 0] >= 0:
                k = acc[b] - 1
                assert (tok[b, :k] == pend_h[b, :k]).all()
                assert (am[b, :k] == pend_h[b, :k]).all()   # accepted = argmax of its anchor
                assert tok[b, k] == am[b, k]                 # replacement / bonus = argmax
            else:
                assert acc[b] == 1 and tok[b, 0] == am[b, N - 1]
        prev = dev
    assert st.diag.cpu().numpy()[isd.DIAG_STATUS] == 0


@pytest.mark.parametrize("greedy", [isd.ISD_SAMPLE, isd.ISD_GREEDY, isd.ISD_ARGMAX_PROPOSE])
def test_rejecting_sequence_ignores_its_draw_rows(greedy):
    """After a rejection the proposals are discarded, so the step does not read the
    sequence's anchor row N-1 and MASK rows: unusable values there change nothing.  A
    sequence that keeps its pending token (q tiny) reads them and fails."""
    N, V = 2, 512
    rng = np.random.default_rng(11)
    host = rng.standard_normal((2, 3, V)).astype(np.float32)
    prev = rng.standard_normal((2, 3, V)).astype(np.float32)
    x0 = int(np.argmin(host[0, 0]))
    host[0, 0, x0] = -np.inf                  # seq 0: p(x) = 0 and x not the argmax: rejected
    x1 = int(np.argmax(host[1, 0]))           # seq 1: the argmax, q tiny: kept
    host[:, 1, 7] = np.nan                    # both sequences' anchor row N-1 ...
    host[:, 2, 3] = np.inf                    # ... and MASK row
    pend, pq = [[x0], [x1]], [[0.5], [1e-30]]
    acc, tok, nq, diag = _one_step(host, prev, pend, pq, N, 1.0, greedy)
    ref = oracle.isd_step(host, prev, pend, pq, N, 1.0, greedy, 5, 0, dtype="f32")
    assert ref["seq_status"].tolist() == [oracle.SEQ_OK, oracle.SEQ_NONFINITE]
    assert acc.tolist() == ref["accepted_len"].tolist() == [1, 0]
    assert (tok == ref["tokens_out"]).all()
    assert diag[isd.DIAG_STATUS] == isd.ISD_ERR_NONFINITE
