"""The step's bounded device waits, made to run out on purpose (no fault, no hang).

isd_debug_set_wait_limit_ns shortens every bounded wait of the step's kernels (the
waits for bulk copies to land) to about a nanosecond.  At B=64, N=4, V=151936 the
statistics pass starts some 20 MB of copies at once, so most warps find their first
copy not yet landed: they give up, report ISD_ERR_TIMEOUT in diag, let their copies in
flight land and leave; the decision pass carries on without the data and still
reaches every cluster barrier.  The call must return and the stream stay usable; once
the workspace is zero-filled again, the same step must give exactly what it gives on a
fresh workspace (the kernels are deterministic).
"""
import numpy as np
import pytest
import torch

from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream
from parity import to_device

pytestmark = pytest.mark.gpu


def _step(st, cur, prev, pend, pq, N, seed, step):
    acc, tok, nq = st.outputs()
    diag = torch.zeros(isd.DIAG_WORDS, dtype=torch.int32, device="cuda")
    isd.isd_step(cur, prev, pend, pq, N, 1.0, False, seed, step, acc, tok, nq, st.p_out, diag, st.workspace)
    torch.cuda.synchronize()
    return diag, [t.cpu().numpy().copy() for t in (acc, tok, nq, st.p_out)]


def test_wait_runs_out_then_the_next_step_is_correct():
    B, N, V = 64, 4, 151936
    gen = ForwardStream(B, N, V, 2.0, 0.5, 3, "bf16")
    h0, h1 = gen.next(), gen.next()
    d0, d1 = to_device(h0, "bf16"), to_device(h1, "bf16")
    st = isd.StepState(B, N, V)
    st.step(d0, None, 1.0, False, 11)        # a first step: pending tokens for the next one
    torch.cuda.synchronize()
    pend, pq = st.pending()
    pend, pq = pend.clone(), pq.clone()
    assert (pend[:, 0] >= 0).any()
    try:
        isd.isd_debug_set_wait_limit_ns(1)
        diag, _ = _step(st, d1, d0, pend, pq, N, 11, 1)   # the call ends: nothing hangs
    finally:
        isd.isd_debug_set_wait_limit_ns(0)
    assert int(diag[isd.DIAG_STATUS].item()) == isd.ISD_ERR_TIMEOUT
    # the context is usable; a zero-filled workspace and the default limit give the step that
    # a fresh workspace gives
    isd.isd_workspace_init(st.workspace)
    diag, got = _step(st, d1, d0, pend, pq, N, 11, 1)
    assert int(diag[isd.DIAG_STATUS].item()) == 0
    fresh = isd.StepState(B, N, V)
    diag2, want = _step(fresh, d1, d0, pend, pq, N, 11, 1)
    assert int(diag2[isd.DIAG_STATUS].item()) == 0
    for g, w, name in zip(got, want, ("accepted_len", "tokens_out", "new_q", "p_out")):
        np.testing.assert_array_equal(g, w, err_msg=name)
