"""The step's bounded device waits, made to run out on purpose (no fault, no hang).

isd_debug_set_wait_limit_ns shortens every bounded wait of the step's kernels (the
waits for bulk copies to land) to about a nanosecond: a warp that finds its copy not
yet landed gives up at once, reports ISD_ERR_TIMEOUT in diag, lets its copies in
flight land and leaves (the statistics pass) or carries on without the data (the
decision pass, which still reaches every cluster barrier).  The call must
return, the stream must stay usable, and after the workspace is zero-filled again a
normal step must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream
from parity import ParityStats, compare_step, to_device

pytestmark = pytest.mark.gpu


def test_wait_runs_out_then_the_next_step_is_correct():
    B, N, V = 4, 4, 4096
    gen = ForwardStream(B, N, V, 2.0, 0.5, 3, "bf16")
    h0, h1 = gen.next(), gen.next()
    d0, d1 = to_device(h0, "bf16"), to_device(h1, "bf16")
    st = isd.StepState(B, N, V)
    st.step(d0, None, 1.0, False, 11)        # a first step: pending tokens for the next one
    torch.cuda.synchronize()
    pend, pq = st.pending()
    pend_h, pq_h = pend.cpu().numpy().copy(), pq.cpu().numpy().copy()
    assert (pend_h[:, 0] >= 0).any()
    acc, tok, nq = st.outputs()
    diag = torch.zeros(isd.DIAG_WORDS, dtype=torch.int32, device="cuda")
    try:
        isd.isd_debug_set_wait_limit_ns(1)
        isd.isd_step(d1, d0, pend, pq, N, 1.0, False, 11, 1, acc, tok, nq, st.p_out, diag, st.workspace)
        torch.cuda.synchronize()             # the call ends: nothing hangs
    finally:
        isd.isd_debug_set_wait_limit_ns(0)
    assert int(diag[isd.DIAG_STATUS].item()) == isd.ISD_ERR_TIMEOUT
    # the context is usable; a zero-filled workspace and the default limit give a correct step
    isd.isd_workspace_init(st.workspace)
    diag.zero_()
    isd.isd_step(d1, d0, pend, pq, N, 1.0, False, 11, 1, acc, tok, nq, st.p_out, diag, st.workspace)
    torch.cuda.synchronize()
    assert int(diag[isd.DIAG_STATUS].item()) == 0
    ref = oracle.isd_step(h1, h0, pend_h, pq_h, N, 1.0, False, 11, 1)
    gpu = dict(accepted_len=acc.cpu().numpy(), tokens_out=tok.cpu().numpy(), new_q=nq.cpu().numpy(),
               p_out=st.p_out.cpu().numpy())
    compare_step(gpu, ref, pend_h, pq_h, N, False, 1.0, h1, h0, 11, 1, "bf16", ParityStats())
