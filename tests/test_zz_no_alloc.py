"""isd_step_noalloc, the entry point for callers that cannot allocate device memory.

Such a caller (for example a plug-in in a host runtime that owns the device memory
and passes only input and output buffers) cannot provide a workspace; the entry
point uses the library's static device scratch instead.  Here it must give the
same outputs as isd_step with a caller-allocated workspace, on two consecutive
steps, the second carrying the first one's proposals.

This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream

pytestmark = pytest.mark.gpu

PROB_RTOL = 1e-5


def _to_device(host, dtype):
    if dtype == "bf16":
        return torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(host)).cuda()


def _two_steps(B, N, V, dtype, T, greedy, use_noalloc, seed):
    gen = ForwardStream(B, N, V, 3.0, 0.5, seed, dtype)
    code = isd.ISD_BF16 if dtype == "bf16" else isd.ISD_F32
    R = 2 * N - 1
    pend = torch.full((B, N - 1), -1, dtype=torch.int32, device="cuda")
    pq = torch.zeros((B, N - 1), dtype=torch.float32, device="cuda")
    ws = None if use_noalloc else isd.alloc_workspace(B, N, V, code)
    diag = torch.zeros(isd.DIAG_WORDS, dtype=torch.int32, device="cuda")
    prev = None
    outs = []
    for t in range(2):
        logits = _to_device(gen.next(), dtype)
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        tok = torch.zeros((B, R), dtype=torch.int32, device="cuda")
        nq = torch.zeros((B, N - 1), dtype=torch.float32, device="cuda")
        pout = torch.zeros((B, N - 1), dtype=torch.float32, device="cuda")
        if use_noalloc:
            isd.isd_step_noalloc(logits, prev, pend, pq, N, T, greedy, 77, t, acc, tok, nq, pout, diag)
        else:
            isd.isd_step(logits, prev, pend, pq, N, T, greedy, 77, t, acc, tok, nq, pout, diag, ws)
        torch.cuda.synchronize()
        outs.append(tuple(x.cpu().numpy().copy() for x in (acc, tok, nq, pout)))
        pend, pq, prev = tok[:, N:], nq, logits
    assert int(diag[isd.DIAG_STATUS]) == 0
    return outs, diag.cpu().numpy()


@pytest.mark.parametrize("B,N,V,dtype,T,greedy", [
    (8, 4, 151936, "bf16", 1.0, False),
    (8, 4, 151936, "bf16", 1.0, True),
    (5, 3, 3000, "f32", 0.7, False),
])
def test_noalloc_matches_isd_step(B, N, V, dtype, T, greedy):
    ref, ref_diag = _two_steps(B, N, V, dtype, T, greedy, False, seed=B + N)
    got, got_diag = _two_steps(B, N, V, dtype, T, greedy, True, seed=B + N)
    for t, (r, g) in enumerate(zip(ref, got)):
        assert (g[0] == r[0]).all(), ("accepted_len", t)
        assert (g[1] == r[1]).all(), ("tokens_out", t)
        np.testing.assert_allclose(g[2], r[2], rtol=PROB_RTOL, atol=0, err_msg="new_q step %d" % t)
        np.testing.assert_allclose(g[3], r[3], rtol=PROB_RTOL, atol=0, err_msg="p_out step %d" % t)
    assert (got_diag == ref_diag).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    B, N, V = 8192, 4, 151936
    assert isd.isd_workspace_size(B, N, V) > isd.STATIC_SCRATCH_BYTES
    logits = torch.empty((1, 2 * N - 1, 8), dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    vp = isd.ctypes.c_void_p
    rc = isd.lib().isd_step_noalloc(vp(logits.data_ptr()), None, isd.ISD_BF16, vp(dummy.data_ptr()), N - 1,
                                    vp(dummy.data_ptr()), B, N, V, 1.0, 0, 0, 0, vp(dummy.data_ptr()),
                                    vp(dummy.data_ptr()), vp(dummy.data_ptr()), None, None, None)
    assert rc == isd.ISD_ERR_SCRATCH_LIMIT
