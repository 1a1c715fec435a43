"""isd_step_fused (the step as one persistent kernel) vs the fp64 oracle, element by element,
under the same parity rule as isd_step (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
from diffusion_lm_decoding_isd_b300 import isd
from oracle.parallel import OraclePool
from parity import check_flag_rate, run_parity, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    """The oracle over the host cores (spawned worker processes)."""
    with OraclePool() as p:
        yield p


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
    stats, diag = run_parity(B, N, V, dtype, 2.0, sigma_n, T, greedy, steps=12, seed=B * 7 + N, fused=True)
    check_flag_rate(stats, V)


@pytest.mark.parametrize("greedy,temperature", [(True, 1.0), (False, 0.7), (isd.ISD_ARGMAX_PROPOSE, 1.0)])
def test_b64_n4_full_vocab(greedy, temperature, pool):
    # B=64, N=4, V=151936 bf16, 16 consecutive steps of each mode
    stats, diag = run_parity(64, 4, 151936, "bf16", 3.0, 0.5, temperature, greedy, steps=16, seed=2, pool=pool,
                             fused=True)
    check_flag_rate(stats, 151936)


def test_b8_n4_full_vocab(pool):
    # B=8, N=4, V=151936 bf16 N(0, 3^2), anchors + N(0, 0.5^2), T=1, 64 steps
    stats, diag = run_parity(8, 4, 151936, "bf16", 3.0, 0.5, 1.0, False, steps=64, seed=1, pool=pool, fused=True)
    check_flag_rate(stats, 151936)
    assert 0.6 < stats.accepts / stats.tests < 0.95
    assert diag[isd.DIAG_RESIDUALS] > 0


def test_q_row_statistics_reread_when_not_chained():
    """Step numbers that skip: every residual streams its q row before its own halves."""
    stats, diag = run_parity(8, 4, 151936, "bf16", 3.0, 0.5, 1.0, False, steps=12, seed=4,
                             step_of=lambda t: 3 * t + 1, fused=True)
    check_flag_rate(stats, 151936)
    assert diag[isd.DIAG_RESIDUALS] > 0


def test_large_vocabulary(pool):
    """1.1 M entries: 538 chunks per row and 1076 residual half chunks."""
    stats, diag = run_parity(8, 2, 1_100_000, "bf16", 3.0, 1.0, 1.0, False, steps=6, seed=9, pool=pool, fused=True)
    check_flag_rate(stats, 1_100_000)
    assert diag[isd.DIAG_RESIDUALS] > 0


def test_many_sequences_small_vocab():
    stats, diag = run_parity(3000, 4, 64, "bf16", 2.0, 0.5, 1.0, False, steps=4, seed=5, fused=True)
    check_flag_rate(stats, 64)


def _one_step(host, prev_host, pend, pq, N, T, greedy):
    B, R, V = host.shape
    dev = to_device(host, "f32")
    prev = None if prev_host is None else to_device(prev_host, "f32")
    st = isd.StepState(B, N, V, isd.ISD_F32, fused=True)
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
        ref = oracle.isd_step(host, prev, pend, pq, N, 1.0, greedy, 5, 0, dtype="f32")
        assert ref["seq_status"].tolist() == [0, 1, 0, 1]
        assert acc.tolist() == ref["accepted_len"].tolist()
        assert (tok == ref["tokens_out"]).all()
        assert diag[isd.DIAG_STATUS] == isd.ISD_ERR_NONFINITE
    acc, tok, nq, diag = _one_step(host[:1], prev[:1], [[V]], [[0.5]], N, 1.0, False)
    assert acc[0] == 0 and diag[isd.DIAG_STATUS] == isd.ISD_ERR_BAD_PENDING
    acc, tok, nq, diag = _one_step(host[:1], prev[:1], [[2]], [[0.0]], N, 1.0, False)
    assert acc[0] == 0 and diag[isd.DIAG_STATUS] == isd.ISD_ERR_BAD_PENDING


@pytest.mark.parametrize("greedy", [isd.ISD_SAMPLE, isd.ISD_GREEDY, isd.ISD_ARGMAX_PROPOSE])
def test_rejecting_sequence_ignores_its_draw_rows(greedy):
    """A rejection discards the proposals, so unusable values in the sequence's anchor row N-1
    and MASK rows change nothing; a sequence that keeps its pending token reads them and fails."""
    N, V = 2, 512
    rng = np.random.default_rng(11)
    host = rng.standard_normal((2, 3, V)).astype(np.float32)
    prev = rng.standard_normal((2, 3, V)).astype(np.float32)
    x0 = int(np.argmin(host[0, 0]))
    host[0, 0, x0] = -np.inf
    x1 = int(np.argmax(host[1, 0]))
    host[:, 1, 7] = np.nan
    host[:, 2, 3] = np.inf
    pend, pq = [[x0], [x1]], [[0.5], [1e-30]]
    acc, tok, nq, diag = _one_step(host, prev, pend, pq, N, 1.0, greedy)
    ref = oracle.isd_step(host, prev, pend, pq, N, 1.0, greedy, 5, 0, dtype="f32")
    assert ref["seq_status"].tolist() == [oracle.SEQ_OK, oracle.SEQ_NONFINITE]
    assert acc.tolist() == ref["accepted_len"].tolist() == [1, 0]
    assert (tok == ref["tokens_out"]).all()
    assert diag[isd.DIAG_STATUS] == isd.ISD_ERR_NONFINITE


def test_one_launch_per_step():
    B, N, V = 4, 4, 4096
    st = isd.StepState(B, N, V, fused=True)
    x = torch.randn((B, 2 * N - 1, V), device="cuda").to(torch.bfloat16)
    st.step(x, None, 1.0, isd.ISD_GREEDY, 0)
    torch.cuda.synchronize()
    assert isd.last_launch_count() == 1
