"""The native library builds, loads, exports the C ABI and checks arguments on the host.

No GPU needed: argument checks return before any CUDA call.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from diffusion_lm_decoding_isd_b300 import build as lib_build
from diffusion_lm_decoding_isd_b300 import isd
from diffusion_lm_decoding_isd_b300.synthetic import (ForwardStream, bf16_bits_to_f32,
                                                      f32_to_bf16_bits, rotating_pool)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return isd.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(isd_\w+)\s*\(", text, flags=re.M):
                names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"isd_step", "isd_workspace_size", "isd_workspace_init", "isd_status_string"} <= names
    for n in names:
        assert hasattr(L, n), n


def test_workspace_size(L):
    assert isd.isd_workspace_size(64, 4, 151936) > 64 * 7 * 75 * 8
    assert isd.isd_workspace_size(1, 2, 1) > 0
    assert isd.isd_workspace_size(0, 4, 100) == 0
    assert isd.isd_workspace_size(4, 1, 100) == 0
    assert isd.isd_workspace_size(4, 33, 100) == 0
    assert isd.isd_workspace_size(4, 4, 0) == 0
    assert isd.isd_workspace_size(4, 4, 100, 7) == 0


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert isd.status_string(code)
    assert isd.status_string(-3).startswith("non-finite")


def _call(L, **kw):
    args = dict(logits=16, prev=16, dtype=0, pend=16, ld=3, pq=16, B=2, N=4, V=128, T=1.0,
                greedy=0, seed=0, step=0, acc=16, tok=16, nq=16, pout=0, diag=0, ws=0, wsb=0,
                stream=0)
    args.update(kw)
    vp = ctypes.c_void_p
    return L.isd_step(vp(args["logits"]), vp(args["prev"]), args["dtype"], vp(args["pend"]),
                      args["ld"], vp(args["pq"]), args["B"], args["N"], args["V"], args["T"],
                      args["greedy"], args["seed"], args["step"], vp(args["acc"]), vp(args["tok"]),
                      vp(args["nq"]), vp(args["pout"]), vp(args["diag"]), vp(args["ws"]),
                      args["wsb"], vp(args["stream"]))


def test_host_argument_checks(L):
    need = isd.isd_workspace_size(2, 4, 128)
    ok_ws = dict(ws=256 * 1000, wsb=need)
    assert _call(L, B=0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, N=1, ld=0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, N=33, ld=32, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, V=0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, dtype=5, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, logits=0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, pend=0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, ld=2, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, T=0.0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, T=float("nan"), **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L, pq=0, **ok_ws) == isd.ISD_ERR_INVALID_ARG
    assert _call(L) == isd.ISD_ERR_WORKSPACE
    assert _call(L, ws=256 * 1000, wsb=need - 1) == isd.ISD_ERR_WORKSPACE
    assert _call(L, ws=256 * 1000 + 16, wsb=need) == isd.ISD_ERR_WORKSPACE
    # greedy mode does not need pending_q nor a temperature
    assert _call(L, greedy=1, pq=0, T=0.0) == isd.ISD_ERR_WORKSPACE


def test_fused_workspace_and_host_argument_checks(L):
    """isd_step_fused: its workspace holds isd_step's sections and its own; the host checks
    are isd_step's, against the larger size."""
    need = isd.isd_fused_workspace_size(2, 4, 128)
    assert need > isd.isd_workspace_size(2, 4, 128)
    # its own sections at B=64, N=4, V=151936: at least the chunk statistics [B][2N-1][C] again
    assert (isd.isd_fused_workspace_size(64, 4, 151936) - isd.isd_workspace_size(64, 4, 151936)
            >= 64 * 7 * 75 * 8)
    for bad in ((0, 4, 100), (4, 1, 100), (4, 33, 100), (4, 4, 0)):
        assert isd.isd_fused_workspace_size(*bad) == 0
    assert isd.isd_fused_workspace_size(4, 4, 100, 7) == 0
    vp = ctypes.c_void_p

    def call(B=2, N=4, V=128, ws=256 * 1000, wsb=need, T=1.0, pq=16, greedy=0):
        return L.isd_step_fused(vp(16), vp(16), 0, vp(16), N - 1, vp(pq), B, N, V, T, greedy, 0, 0,
                                vp(16), vp(16), vp(16), vp(0), vp(0), vp(ws), wsb, vp(0))
    assert call(B=0) == isd.ISD_ERR_INVALID_ARG
    assert call(N=1) == isd.ISD_ERR_INVALID_ARG
    assert call(T=0.0) == isd.ISD_ERR_INVALID_ARG
    assert call(pq=0) == isd.ISD_ERR_INVALID_ARG
    assert call(greedy=3) == isd.ISD_ERR_INVALID_ARG
    assert call(ws=0) == isd.ISD_ERR_WORKSPACE
    assert call(wsb=isd.isd_workspace_size(2, 4, 128)) == isd.ISD_ERR_WORKSPACE  # isd_step's size is too small
    assert call(wsb=need - 1) == isd.ISD_ERR_WORKSPACE
    assert call(ws=256 * 1000 + 16) == isd.ISD_ERR_WORKSPACE
    assert L.isd_last_launch_count() == 0


def test_bf16_rounding_matches_definition():
    x = np.array([1.0, 1.00390625, 1.005859375, -np.inf, 3.14159, -2.5e-3, 0.0, -0.0],
                 dtype=np.float32)
    b = f32_to_bf16_bits(x)
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F81, 0xFF80, 0x4049, 0xBB24, 0x0000, 0x8000]
    assert (bf16_bits_to_f32(b)[[0, 3]] == np.array([1.0, -np.inf], dtype=np.float32)).all()


def test_forward_stream_relation():
    B, N, V = 3, 4, 64
    g = ForwardStream(B, N, V, 3.0, 0.5, 0, "f32")
    a = g.next()
    b = g.next()
    d = b[:, :N - 1] - a[:, N:]
    assert abs(d.std() - 0.5) < 0.1 and abs(a.std() - 3.0) < 0.3


def test_rotating_pool_is_circular():
    B, N, V = 2, 3, 32
    bufs = rotating_pool(B, N, V, 3.0, 0.0, 1, 3, "bf16")
    for k in range(3):
        assert (bufs[k][:, :N - 1] == bufs[k - 1][:, N:]).all()


def test_lm_head_host_argument_checks(L):
    vp = ctypes.c_void_p
    call = lambda h=16, w=16, M=4, K=64, V=128, out=16: L.isd_lm_head(vp(h), vp(w), M, K, V, vp(out), vp(0), vp(0))
    assert call(h=0) == isd.ISD_ERR_INVALID_ARG
    assert call(out=0) == isd.ISD_ERR_INVALID_ARG
    assert call(M=0) == isd.ISD_ERR_INVALID_ARG
    assert call(K=12) == isd.ISD_ERR_INVALID_ARG      # rows must be 16-byte multiples
    assert call(K=0) == isd.ISD_ERR_INVALID_ARG
    assert call(V=0) == isd.ISD_ERR_INVALID_ARG
    assert call(h=24) == isd.ISD_ERR_INVALID_ARG      # 16-byte alignment
    assert L.isd_lm_head_last_launch_count() == 0


def test_from_hidden_host_argument_checks(L):
    vp = ctypes.c_void_p
    need = isd.isd_from_hidden_workspace_size(2, 4, 128)
    assert need > isd.isd_workspace_size(2, 4, 128)
    assert isd.isd_from_hidden_workspace_size(0, 4, 128) == 0

    def call(B=2, N=4, V=128, K=64, ws=256 * 1000, wsb=need, T=1.0, pq=16):
        return L.isd_step_from_hidden(vp(16), vp(16), K, vp(16), vp(16), vp(16), N - 1, vp(pq), B, N, V,
                                      T, 0, 0, 0, vp(16), vp(16), vp(16), vp(0), vp(0), vp(ws), wsb, vp(0))
    assert call(B=0) == isd.ISD_ERR_INVALID_ARG
    assert call(N=1) == isd.ISD_ERR_INVALID_ARG
    assert call(K=10) == isd.ISD_ERR_INVALID_ARG
    assert call(T=0.0) == isd.ISD_ERR_INVALID_ARG
    assert call(pq=0) == isd.ISD_ERR_INVALID_ARG
    assert call(wsb=need - 1) == isd.ISD_ERR_WORKSPACE
    assert call(ws=256 * 1000 + 8) == isd.ISD_ERR_WORKSPACE


def test_derived_tpf_metrics_match_the_pages_figures():
    import bench
    # N=4, p=0.9: TPF 2.919 (closed form), efficiency TPF^2/7 = 1.217, R-ISD speedup TPF/1.12 = 2.606
    tpf = bench.tpf_closed_form(0.9, 4)
    d = bench.derived_tpf_metrics(tpf, 4)
    assert abs(tpf - 2.919) < 1e-3
    assert abs(d["compute_efficiency"] - 1.217) < 1e-3
    assert abs(d["r_isd_speedup"] - 2.606) < 1e-3


def test_binding_rejects_host_tensors_before_any_call():
    """The binding checks layouts on the host and raises before the library is called."""
    import torch
    h = torch.zeros((4, 64), dtype=torch.bfloat16)
    w = torch.zeros((8, 64), dtype=torch.bfloat16)
    out = torch.zeros((4, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        isd.isd_lm_head(h, w, out)  # CPU tensors
    logits = torch.zeros((2, 7, 8), dtype=torch.bfloat16)
    pend = torch.zeros((2, 3), dtype=torch.int32)
    with pytest.raises(ValueError):
        isd.isd_step(logits, None, pend, None, 3, 1.0, True, 0, 0, torch.zeros(2, dtype=torch.int32),
                     torch.zeros((2, 7), dtype=torch.int32), torch.zeros((2, 3)), workspace=None)


def test_source_code_hash_ignores_comments(tmp_path):
    import bench
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text("int f() {  // one\n    return 1;\n}\n")
    b.write_text("// header\nint f() {  // another comment\n\n    return 1;\n}\n")
    assert bench.source_code_hash(str(a)) == bench.source_code_hash(str(b))
    b.write_text("int f() {\n    return 2;\n}\n")
    assert bench.source_code_hash(str(a)) != bench.source_code_hash(str(b))
    # a record over several files changes when any of them does
    c = tmp_path / "c.cuh"
    c.write_text("int g();\n")
    h = bench.sources_code_hash([str(a), str(c)])
    assert h == bench.sources_code_hash([str(a), str(c)])
    c.write_text("int g(); // only a comment more\n")
    assert h == bench.sources_code_hash([str(a), str(c)])
    c.write_text("int g(int);\n")
    assert h != bench.sources_code_hash([str(a), str(c)])


def test_mode_constants_match_the_header():
    text = open(os.path.join(ROOT, "include", "isd.h")).read()
    assert re.search(r"ISD_SAMPLE = 0", text) and re.search(r"ISD_GREEDY = 1", text)
    assert re.search(r"ISD_ARGMAX_PROPOSE = 2", text)
    assert (isd.ISD_SAMPLE, isd.ISD_GREEDY, isd.ISD_ARGMAX_PROPOSE) == (0, 1, 2)


def test_byte_accounting_of_the_benchmark():
    """The roofline's bytes: the statistics pass reads rows N-1..2N-2 of every sequence and the
    N-1 anchor rows of every sequence with pending tokens; the method's own bytes count the
    rows its decisions read, the residual's two rows and one chunk per draw."""
    import bench
    B, N, V, esz, steps = 64, 4, 151936, 2, 10
    recovery = 290                     # sequence-steps without pending tokens
    pending = steps * B - recovery
    assert bench.stats_pass_bytes(steps, B, N, V, esz, recovery) == (steps * B * N + pending * (N - 1)) * V * esz
    assert bench.stats_pass_bytes(1, 1, 2, 8, 4, 1) == 2 * 8 * 4  # no pending tokens: rows N-1, N only
    tests, accepts = 700, 560          # 140 rejections
    rejecting = tests - accepts
    proposing = steps * B - rejecting
    row = V * esz
    want = (pending * (N - 1) + proposing * N + 2 * rejecting) * row + (proposing * N + rejecting) * bench.CHUNK_BYTES
    assert bench.step_bytes(steps, B, N, V, esz, 0, recovery, tests, accepts) == want
    # greedy: no residual rows, no draws that read a chunk again
    want_g = (pending * (N - 1) + proposing * N) * row
    assert bench.step_bytes(steps, B, N, V, esz, 1, recovery, tests, accepts) == want_g
