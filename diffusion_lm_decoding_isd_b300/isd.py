"""Thin ctypes binding of the C ABI in include/isd.h (same names, argument marshalling only).

Tensors are PyTorch CUDA tensors (PyTorch provides device memory and streams);
every step of the computation runs in the native library's CUDA kernels.  If the
library is missing the first call raises: there is no fallback.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libisd_b300.so")

ISD_OK = 0
ISD_ERR_INVALID_ARG = -1
ISD_ERR_CUDA = -2
ISD_ERR_NONFINITE = -3
ISD_ERR_WORKSPACE = -4
ISD_ERR_TIMEOUT = -5
ISD_ERR_BAD_PENDING = -6
ISD_ERR_SCRATCH_LIMIT = -7
STATIC_SCRATCH_BYTES = 8 << 20

ISD_BF16 = 0
ISD_F32 = 1

DIAG_STATUS, DIAG_ACCEPTS, DIAG_TESTS, DIAG_NEAR_TIE_ACC, DIAG_NEAR_TIE_CDF = 0, 1, 2, 3, 4
DIAG_RESIDUALS, DIAG_RECOVERY, DIAG_EMITTED, DIAG_WORDS = 5, 6, 7, 8
MAX_N = 32
ISD_SAMPLE, ISD_GREEDY, ISD_ARGMAX_PROPOSE = 0, 1, 2

_lib = None


class ISDError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s: %s (%d)" % (what, status_string(code) if _lib else "?", code))
        self.code = code


def lib():
    """The loaded native library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("native library %s is missing; build it with "
                               "`python -m diffusion_lm_decoding_isd_b300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
        L.isd_workspace_size.argtypes = [i32, i32, i32, i32]
        L.isd_workspace_size.restype = sz
        L.isd_workspace_init.argtypes = [vp, sz, vp]
        L.isd_workspace_init.restype = i32
        L.isd_step.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, f32, i32, u64, u64,
                               vp, vp, vp, vp, vp, vp, sz, vp]
        L.isd_step.restype = i32
        L.isd_step_noalloc.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, f32, i32, u64, u64,
                                       vp, vp, vp, vp, vp, vp]
        L.isd_step_noalloc.restype = i32
        L.isd_fused_workspace_size.argtypes = [i32, i32, i32, i32]
        L.isd_fused_workspace_size.restype = sz
        L.isd_step_fused.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, f32, i32, u64, u64,
                                     vp, vp, vp, vp, vp, vp, sz, vp]
        L.isd_step_fused.restype = i32
        L.isd_lm_head.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
        L.isd_lm_head.restype = i32
        L.isd_from_hidden_workspace_size.argtypes = [i32, i32, i32]
        L.isd_from_hidden_workspace_size.restype = sz
        L.isd_lm_head_last_launch_count.argtypes = []
        L.isd_lm_head_last_launch_count.restype = i32
        L.isd_step_from_hidden.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, i32, i32, i32, f32, i32, u64, u64,
                                           vp, vp, vp, vp, vp, vp, sz, vp]
        L.isd_step_from_hidden.restype = i32
        L.isd_status_string.argtypes = [i32]
        L.isd_status_string.restype = ctypes.c_char_p
        L.isd_last_launch_count.argtypes = []
        L.isd_last_launch_count.restype = i32
        L.isd_profile_begin.argtypes = [i32]
        L.isd_profile_begin.restype = i32
        L.isd_profile_read.argtypes = [i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32)]
        L.isd_profile_read.restype = i32
        L.isd_profile_end.argtypes = []
        L.isd_profile_end.restype = None
        L.isd_debug_set_wait_limit_ns.argtypes = [u64]
        L.isd_debug_set_wait_limit_ns.restype = i32
        _lib = L
    return _lib


def status_string(code):
    return lib().isd_status_string(int(code)).decode()


def dtype_code(t):
    if t.dtype == torch.bfloat16:
        return ISD_BF16
    if t.dtype == torch.float32:
        return ISD_F32
    raise TypeError("logits must be bfloat16 or float32")


def isd_workspace_size(B, N, V, dtype=ISD_BF16):
    return int(lib().isd_workspace_size(int(B), int(N), int(V), int(dtype)))


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def isd_from_hidden_workspace_size(B, N, V):
    return int(lib().isd_from_hidden_workspace_size(int(B), int(N), int(V)))


def isd_fused_workspace_size(B, N, V, dtype=ISD_BF16):
    return int(lib().isd_fused_workspace_size(int(B), int(N), int(V), int(dtype)))


def alloc_workspace(B, N, V, dtype=ISD_BF16, device="cuda", stream=None, from_hidden=False, fused=False):
    """Allocate (through PyTorch) and zero-fill a workspace for these sizes (for
    isd_step_from_hidden if from_hidden, for isd_step_fused if fused)."""
    if from_hidden and fused:
        raise ValueError("a workspace serves isd_step_from_hidden or isd_step_fused, not both")
    if from_hidden:
        n = isd_from_hidden_workspace_size(B, N, V)
    elif fused:
        n = isd_fused_workspace_size(B, N, V, dtype)
    else:
        n = isd_workspace_size(B, N, V, dtype)
    if n == 0:
        raise ValueError("unsupported sizes B=%d N=%d V=%d" % (B, N, V))
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    isd_workspace_init(ws, stream)
    return ws


def isd_workspace_init(workspace, stream=None):
    rc = lib().isd_workspace_init(ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                  _stream_ptr(stream))
    if rc != ISD_OK:
        raise ISDError(rc, "isd_workspace_init")


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def isd_step(logits, prev_logits, pending_tokens, pending_q, N, temperature, greedy,
             philox_seed, step, accepted_len, tokens_out, new_q, p_out=None, diag=None,
             workspace=None, stream=None, check=True):
    """One ISD verify-and-propose step (see include/isd.h).  All tensors are CUDA
    tensors in the layouts the header states; outputs are written in place.
    pending_tokens may be a [B][N-1] view with unit inner stride (e.g. the
    previous step's tokens_out[:, N:]); its row stride becomes pending_ld.
    greedy: ISD_SAMPLE (0 / False), ISD_GREEDY (1 / True) or ISD_ARGMAX_PROPOSE (2)."""
    B, R, V = logits.shape
    if R != 2 * N - 1:
        raise ValueError("logits must be [B][2N-1][V]")
    for name, t in (("logits", logits), ("accepted_len", accepted_len),
                    ("tokens_out", tokens_out), ("new_q", new_q)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if (not pending_tokens.is_cuda or pending_tokens.dtype != torch.int32
            or tuple(pending_tokens.shape) != (B, N - 1) or pending_tokens.stride(1) != 1):
        raise ValueError("pending_tokens must be an int32 CUDA [B][N-1] view with unit inner stride")
    dt = dtype_code(logits)
    if prev_logits is not None and (prev_logits.dtype != logits.dtype or prev_logits.shape != logits.shape):
        raise ValueError("prev_logits must match logits")
    if workspace is None:
        raise ValueError("workspace is required (alloc_workspace)")
    rc = lib().isd_step(_ptr(logits), _ptr(prev_logits), dt, _ptr(pending_tokens),
                        int(pending_tokens.stride(0)), _ptr(pending_q),
                        int(B), int(N), int(V), float(temperature), int(greedy),
                        int(philox_seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF,
                        _ptr(accepted_len), _ptr(tokens_out), _ptr(new_q), _ptr(p_out), _ptr(diag),
                        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    if check and rc != ISD_OK:
        raise ISDError(rc, "isd_step")
    return rc


def isd_step_fused(logits, prev_logits, pending_tokens, pending_q, N, temperature, greedy,
                   philox_seed, step, accepted_len, tokens_out, new_q, p_out=None, diag=None,
                   workspace=None, stream=None, check=True):
    """isd_step as one persistent kernel (see include/isd.h, isd_step_fused): the
    same arguments and results; the workspace comes from alloc_workspace(..., fused=True)."""
    B, V = _check_step_args(logits, prev_logits, pending_tokens, N, accepted_len, tokens_out, new_q)
    if workspace is None:
        raise ValueError("workspace is required (alloc_workspace(..., fused=True))")
    rc = lib().isd_step_fused(_ptr(logits), _ptr(prev_logits), dtype_code(logits), _ptr(pending_tokens),
                              int(pending_tokens.stride(0)), _ptr(pending_q),
                              int(B), int(N), int(V), float(temperature), int(greedy),
                              int(philox_seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF,
                              _ptr(accepted_len), _ptr(tokens_out), _ptr(new_q), _ptr(p_out), _ptr(diag),
                              ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    if check and rc != ISD_OK:
        raise ISDError(rc, "isd_step_fused")
    return rc


def _check_step_args(logits, prev_logits, pending_tokens, N, accepted_len, tokens_out, new_q):
    B, R, V = logits.shape
    if R != 2 * N - 1:
        raise ValueError("logits must be [B][2N-1][V]")
    for name, t in (("logits", logits), ("accepted_len", accepted_len),
                    ("tokens_out", tokens_out), ("new_q", new_q)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if (not pending_tokens.is_cuda or pending_tokens.dtype != torch.int32
            or tuple(pending_tokens.shape) != (B, N - 1) or pending_tokens.stride(1) != 1):
        raise ValueError("pending_tokens must be an int32 CUDA [B][N-1] view with unit inner stride")
    if prev_logits is not None and (prev_logits.dtype != logits.dtype or prev_logits.shape != logits.shape):
        raise ValueError("prev_logits must match logits")
    return B, V


def isd_step_noalloc(logits, prev_logits, pending_tokens, pending_q, N, temperature, greedy,
                     philox_seed, step, accepted_len, tokens_out, new_q, p_out=None, diag=None,
                     stream=None, check=True):
    """isd_step with the library's static scratch instead of a workspace (see
    include/isd.h: for callers that cannot allocate device memory; calls that
    overlap on the GPU race on the shared scratch)."""
    B, V = _check_step_args(logits, prev_logits, pending_tokens, N, accepted_len, tokens_out, new_q)
    rc = lib().isd_step_noalloc(_ptr(logits), _ptr(prev_logits), dtype_code(logits), _ptr(pending_tokens),
                                int(pending_tokens.stride(0)), _ptr(pending_q),
                                int(B), int(N), int(V), float(temperature), int(greedy),
                                int(philox_seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF,
                                _ptr(accepted_len), _ptr(tokens_out), _ptr(new_q), _ptr(p_out),
                                _ptr(diag), _stream_ptr(stream))
    if check and rc != ISD_OK:
        raise ISDError(rc, "isd_step_noalloc")
    return rc


def _check_bf16_matrix(name, t, rows=None, cols=None):
    if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or t.dim() != 2:
        raise ValueError("%s must be a contiguous 2-D bf16 CUDA tensor" % name)
    if (rows is not None and t.shape[0] != rows) or (cols is not None and t.shape[1] != cols):
        raise ValueError("%s has shape %s" % (name, tuple(t.shape)))


def isd_lm_head(hidden, lm_head, logits, status=None, stream=None, check=True):
    """logits[M][V] = bf16(hidden[M][K] @ lm_head[V][K]^T), fp32 accumulation on
    the tensor cores (see include/isd.h).  status: optional int32 CUDA tensor."""
    _check_bf16_matrix("hidden", hidden)
    M, K = hidden.shape
    _check_bf16_matrix("lm_head", lm_head, cols=K)
    V = lm_head.shape[0]
    _check_bf16_matrix("logits", logits, rows=M, cols=V)
    rc = lib().isd_lm_head(_ptr(hidden), _ptr(lm_head), int(M), int(K), int(V), _ptr(logits), _ptr(status),
                           _stream_ptr(stream))
    if check and rc != ISD_OK:
        raise ISDError(rc, "isd_lm_head")
    return rc


def isd_step_from_hidden(hidden, lm_head, logits, prev_logits, pending_tokens, pending_q, N, temperature,
                         greedy, philox_seed, step, accepted_len, tokens_out, new_q, p_out=None, diag=None,
                         workspace=None, stream=None, check=True):
    """isd_lm_head into `logits` ([B][2N-1][V] bf16), then isd_step on it.
    hidden is [B][2N-1][K] bf16, lm_head [V][K] bf16."""
    if hidden.dim() != 3 or not hidden.is_cuda or not hidden.is_contiguous() or hidden.dtype != torch.bfloat16:
        raise ValueError("hidden must be a contiguous [B][2N-1][K] bf16 CUDA tensor")
    B, R, K = hidden.shape
    _check_bf16_matrix("lm_head", lm_head, cols=K)
    V = lm_head.shape[0]
    if tuple(logits.shape) != (B, R, V) or logits.dtype != torch.bfloat16:
        raise ValueError("logits must be a [B][2N-1][V] bf16 tensor")
    _check_step_args(logits, prev_logits, pending_tokens, N, accepted_len, tokens_out, new_q)
    if workspace is None:
        raise ValueError("workspace is required (alloc_workspace)")
    rc = lib().isd_step_from_hidden(_ptr(hidden), _ptr(lm_head), int(K), _ptr(logits), _ptr(prev_logits),
                                    _ptr(pending_tokens), int(pending_tokens.stride(0)), _ptr(pending_q),
                                    int(B), int(N), int(V), float(temperature), int(greedy),
                                    int(philox_seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF,
                                    _ptr(accepted_len), _ptr(tokens_out), _ptr(new_q), _ptr(p_out), _ptr(diag),
                                    ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    if check and rc != ISD_OK:
        raise ISDError(rc, "isd_step_from_hidden")
    return rc


def lm_head_last_launch_count():
    return int(lib().isd_lm_head_last_launch_count())


def last_launch_count():
    return int(lib().isd_last_launch_count())


KERNEL_STATS, KERNEL_DECIDE, KERNEL_LM_HEAD, KERNEL_MERGE, KERNEL_FUSED = 0, 1, 2, 3, 4
KERNEL_NAMES = {0: "isd_stats_kernel", 1: "isd_decide_kernel", 2: "isd_lm_head_kernel", 3: "isd_lm_head_merge_kernel",
                4: "isd_fused_step_kernel"}


def isd_profile_begin(capacity):
    rc = lib().isd_profile_begin(int(capacity))
    if rc != ISD_OK:
        raise ISDError(rc, "isd_profile_begin")


def isd_profile_read(kind):
    """(total milliseconds, launches) of the recorded kernels of one kind."""
    ms = ctypes.c_double()
    n = ctypes.c_int()
    rc = lib().isd_profile_read(int(kind), ctypes.byref(ms), ctypes.byref(n))
    if rc != ISD_OK:
        raise ISDError(rc, "isd_profile_read")
    return ms.value, n.value


def isd_profile_end():
    lib().isd_profile_end()


def isd_debug_set_wait_limit_ns(ns):
    """Testing hook: how long the step's bounded device waits last before they give up
    (0 restores the default of about one second)."""
    lib().isd_debug_set_wait_limit_ns(int(ns))


class StepState:
    """Carried state and outputs for a batch, double-buffered so that each step
    reads the previous step's proposals in place (pending = tokens_out[:, N:])."""

    def __init__(self, B, N, V, dtype=ISD_BF16, device="cuda", from_hidden=False, fused=False):
        """fused: step() runs isd_step_fused instead of isd_step."""
        R = 2 * N - 1
        self.B, self.N, self.V = B, N, V
        self.fused = fused
        self.start_pending = torch.full((B, N - 1), -1, dtype=torch.int32, device=device)
        self.start_q = torch.zeros((B, N - 1), dtype=torch.float32, device=device)
        self.accepted_len = [torch.zeros(B, dtype=torch.int32, device=device) for _ in range(2)]
        self.tokens_out = [torch.zeros((B, R), dtype=torch.int32, device=device) for _ in range(2)]
        self.new_q = [torch.zeros((B, N - 1), dtype=torch.float32, device=device) for _ in range(2)]
        self.p_out = torch.zeros((B, N - 1), dtype=torch.float32, device=device)
        self.diag = torch.zeros(DIAG_WORDS, dtype=torch.int32, device=device)
        self.workspace = alloc_workspace(B, N, V, dtype, device, from_hidden=from_hidden, fused=fused)
        self.t = 0

    def pending(self):
        if self.t == 0:
            return self.start_pending, self.start_q
        j = (self.t - 1) & 1
        return self.tokens_out[j][:, self.N:], self.new_q[j]

    def outputs(self):
        j = self.t & 1
        return self.accepted_len[j], self.tokens_out[j], self.new_q[j]

    def step(self, logits, prev_logits, temperature, greedy, seed, step=None, stream=None,
             accepted_len=None):
        """Run one isd_step on this state and advance it.  `accepted_len` may name
        another int32 [B] tensor to receive this step's accepted lengths."""
        pend, pq = self.pending()
        acc, tok, nq = self.outputs()
        if accepted_len is not None:
            acc = accepted_len
        fn = isd_step_fused if self.fused else isd_step
        fn(logits, prev_logits, pend, pq, self.N, temperature, greedy, seed,
           self.t if step is None else step, acc, tok, nq, self.p_out, self.diag,
           self.workspace, stream)
        self.t += 1
        return acc, tok, nq

    def step_from_hidden(self, hidden, lm_head, logits, prev_logits, temperature, greedy, seed, step=None,
                         stream=None):
        """isd_step_from_hidden on this state: the projection writes `logits`
        ([B][2N-1][V] bf16, kept for the next step's prev_logits), then the step."""
        pend, pq = self.pending()
        acc, tok, nq = self.outputs()
        isd_step_from_hidden(hidden, lm_head, logits, prev_logits, pend, pq, self.N, temperature, greedy, seed,
                             self.t if step is None else step, acc, tok, nq, self.p_out, self.diag,
                             self.workspace, stream)
        self.t += 1
        return acc, tok, nq
