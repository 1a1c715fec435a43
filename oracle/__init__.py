"""fp64 CPU oracle of the ISD verify-and-propose step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product path never does.

The arithmetic lives in ``isd_oracle.c``; this module marshals numpy arrays to
it through ctypes.  Logits are passed either as ``float32`` arrays or as
``uint16`` arrays holding bf16 bit patterns (``dtype="bf16"``).
"""
import contextlib
import ctypes
import os

import numpy as np

from . import build as _build

DTYPE_BF16 = 0
DTYPE_F32 = 1

SEQ_OK = 0
SEQ_NONFINITE = 1
SEQ_BAD_PENDING = 2

_lib = None


def _load(path=None):
    global _lib
    if _lib is None:
        path = path or _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        fp = ctypes.POINTER(ctypes.c_float)
        up = ctypes.POINTER(ctypes.c_uint32)
        vp = ctypes.c_void_p
        lib.oracle_philox4x32_10.argtypes = [up, up, up]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_uniform.argtypes = [ctypes.c_uint32]
        lib.oracle_uniform.restype = ctypes.c_double
        lib.oracle_row_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                            ctypes.c_uint32, dp, dp]
        lib.oracle_row_uniforms.restype = None
        common = [vp, vp, ctypes.c_int, ip, fp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_double, ctypes.c_int]
        outs = [ip, ip, dp, dp, ip, dp, dp, ctypes.c_double, ip, ip]
        lib.oracle_isd_step_u.argtypes = common + [dp, dp] + outs
        lib.oracle_isd_step_u.restype = ctypes.c_int
        lib.oracle_isd_step.argtypes = common + [ctypes.c_uint64, ctypes.c_uint64] + outs
        lib.oracle_isd_step.restype = ctypes.c_int
        lib.oracle_softmax_prob.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_softmax_prob.restype = ctypes.c_double
        _lib = lib
    return _lib


@contextlib.contextmanager
def using_library(path):
    """Run the block against another build of the oracle (used by the test
    that plants mistakes in a copy of the source)."""
    global _lib
    saved = _lib
    _lib = None
    _load(path)
    try:
        yield
    finally:
        _lib = saved


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def philox4x32_10(ctr, key):
    """Philox4x32-10 of a 4-word counter and 2-word key -> 4 words."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32),
                             _ptr(out, ctypes.c_uint32))
    return [int(x) for x in out]


def uniform(word):
    return _load().oracle_uniform(int(word) & 0xFFFFFFFF)


def row_uniforms(seed, step, seq, row):
    """(u_accept, u_sample) of one logit row."""
    a = ctypes.c_double()
    s = ctypes.c_double()
    _load().oracle_row_uniforms(seed, step, seq, row, ctypes.byref(a), ctypes.byref(s))
    return a.value, s.value


def _logits_arg(x, dtype):
    if x is None:
        return None, None
    if dtype == "bf16":
        arr = np.ascontiguousarray(x, dtype=np.uint16)
    elif dtype == "f32":
        arr = np.ascontiguousarray(x, dtype=np.float32)
    else:
        raise ValueError("dtype must be 'bf16' or 'f32'")
    return arr, ctypes.c_void_p(arr.ctypes.data)


# Half-width of the near-tie window, relative: an acceptance test with
# |u - p/q| below it, or an inverse-CDF draw whose target lies within it times
# the sum of the weights from a CDF edge, is a near-tie.
NEAR_TOL = 1e-6


def _step(fn, extra, logits, prev_logits, pending_tokens, pending_q, N, temperature,
          greedy, dtype, near_tol=NEAR_TOL):
    lib = _load()
    larr, lptr = _logits_arg(logits, dtype)
    parr, pptr = _logits_arg(prev_logits, dtype)
    B, R, V = larr.shape
    assert R == 2 * N - 1, "logits must be [B][2N-1][V]"
    if parr is not None:
        assert parr.shape == larr.shape
    pt = np.ascontiguousarray(np.asarray(pending_tokens, dtype=np.int32).reshape(B, N - 1))
    pq = np.ascontiguousarray(np.asarray(pending_q, dtype=np.float32).reshape(B, N - 1))
    acc = np.zeros(B, dtype=np.int32)
    tok = np.zeros((B, R), dtype=np.int32)
    nq = np.zeros((B, N - 1), dtype=np.float64)
    pout = np.zeros((B, N - 1), dtype=np.float64)
    st = np.zeros(B, dtype=np.int32)
    am = np.zeros((B, N - 1), dtype=np.float64)
    cm = np.zeros((B, R), dtype=np.float64)
    clo = np.zeros((B, R), dtype=np.int32)
    chi = np.zeros((B, R), dtype=np.int32)
    code = DTYPE_BF16 if dtype == "bf16" else DTYPE_F32
    rc = fn(lptr, pptr, code, _ptr(pt, ctypes.c_int32), _ptr(pq, ctypes.c_float),
            B, N, V, float(temperature), int(greedy), *extra(B, R),
            _ptr(acc, ctypes.c_int32), _ptr(tok, ctypes.c_int32), _ptr(nq, ctypes.c_double),
            _ptr(pout, ctypes.c_double), _ptr(st, ctypes.c_int32), _ptr(am, ctypes.c_double),
            _ptr(cm, ctypes.c_double), float(near_tol), _ptr(clo, ctypes.c_int32),
            _ptr(chi, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dict(accepted_len=acc, tokens_out=tok, new_q=nq, p_out=pout, seq_status=st,
                accept_margin=am, cdf_margin=cm, cdf_lo=clo, cdf_hi=chi)


def isd_step(logits, prev_logits, pending_tokens, pending_q, N, temperature, greedy,
             seed, step, dtype="bf16", near_tol=NEAR_TOL):
    """One ISD step for all sequences, uniforms from Philox (seed, step, seq, row).

    Besides the step's outputs, for every inverse-CDF draw made at row r of
    sequence b: cdf_margin[b, r] (distance of the target from the nearer edge
    of the chosen token's interval, relative to the sum of the weights) and
    [cdf_lo[b, r], cdf_hi[b, r]], the tokens whose interval comes within
    near_tol of the target; -1 where no draw was made."""
    lib = _load()
    return _step(lib.oracle_isd_step, lambda B, R: (int(seed), int(step)), logits,
                 prev_logits, pending_tokens, pending_q, N, temperature, greedy, dtype, near_tol)


def isd_step_u(logits, prev_logits, pending_tokens, pending_q, N, temperature, greedy,
               u_accept, u_sample, dtype="bf16", near_tol=NEAR_TOL):
    """One ISD step with the uniforms of every row given ([B][2N-1] each)."""
    lib = _load()
    keep = []

    def extra(B, R):
        a = np.ascontiguousarray(np.asarray(u_accept, dtype=np.float64).reshape(B, R))
        s = np.ascontiguousarray(np.asarray(u_sample, dtype=np.float64).reshape(B, R))
        keep.extend([a, s])
        return _ptr(a, ctypes.c_double), _ptr(s, ctypes.c_double)

    return _step(lib.oracle_isd_step_u, extra, logits, prev_logits, pending_tokens,
                 pending_q, N, temperature, greedy, dtype, near_tol)


def softmax_prob(row, temperature, token, dtype="bf16"):
    """softmax(row / T)[token] in fp64 for one logit row (bf16 bits or fp32)."""
    arr, ptr = _logits_arg(np.ascontiguousarray(row).reshape(-1), dtype)
    p = _load().oracle_softmax_prob(ptr, DTYPE_BF16 if dtype == "bf16" else DTYPE_F32, arr.shape[0],
                                    float(temperature), int(token))
    if p < 0:
        raise ValueError("oracle rejected the arguments")
    return p
