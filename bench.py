#!/usr/bin/env python3
"""Benchmark of the ISD verify-and-propose step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-e2e]
    python bench.py --sweep [--sweep-steps S]

A step is one isd_step over one batch of synthetic forward logits (the default
workload: B=64 sequences, N=4 (7 rows each), V=151936 bf16, sampling at
T=0.7).  Inputs are resident in HBM before timing; four rotating logits buffers
of 136 MB each (each larger than the 126 MB L2) are cycled.  Steps are replayed
from CUDA graphs of up to 32 consecutive steps.  A timed block is exactly
--steps steps between two device synchronisations; blocks are repeated until
about half a second of device time is covered, and the median block gives
ms_per_step (p10 / p90 reported beside it).  The default workload's line also
carries the from-hidden workload (LM-head projection + step) as a nested
object.  Prints one JSON line.

Under torchrun each rank runs its own replica of the workload on its own GPU
(sequences are independent: weak scaling, no collective on the data path);
rank 0 prints the line with the max time over ranks.

--impl reference times the fp64 CPU oracle on the host cores (one sequence of
the workload per step).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tokens/s and logits GB/s (% of HBM peak), B=64 N=4 V=151936, 1 B300"
UNIT = "tokens/s"
N_BUFFERS = 4
FALLBACK_HBM_GBS = 6400.0
NOMINAL_HBM_GBS = 8000.0
DEFAULT_WORKLOAD = "b64_n4_v151936_t0.7"
FROM_HIDDEN_STEPS = 16  # steps per timed block of the nested from-hidden record


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x, world):
    """Max of a host float over all ranks (gloo; no data-path collective)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index, period_ms=20):
        self.dev = device_index
        self.period = period_ms
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + CLOCK_FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(", ") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        return rows


def summarize_clocks(rows, t_rows=None):
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
        except (ValueError, IndexError):
            continue
        for name, val in zip(names, r[5:9]):
            if val.strip().lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------
# replaying steps from CUDA graphs, timed in blocks of exactly K steps
# ------------------------------------------------------------------------------------
PHASES = 4          # steps cycle 4 input buffers and 2 state buffers: index mod 4
MAX_GRAPH_STEPS = 32
MIN_TIMED_MS = 500.0
FUSED_STEPS = 2000  # steps per timed block of the isd_step_fused line


class Replayer:
    """Consecutive steps replayed from CUDA graphs.  A graph bakes in the buffers of the
    steps it captured, so one is captured per (starting phase, length), phase being the
    step index mod 4; a block of K steps is a chain of such graphs.  `step_fn(t)` runs
    step t through `state` (whose counter `t` must equal the argument)."""

    def __init__(self, torch, state, step_fn, dev, max_len=MAX_GRAPH_STEPS):
        self.torch, self.state, self.step_fn, self.max_len = torch, state, step_fn, max_len
        self.cap = torch.cuda.Stream(device=dev)
        self.graphs = {}
        self.pos = state.t  # index of the next step

    def capture(self, phase, length):
        torch = self.torch
        saved = self.state.t
        self.state.t = PHASES * (1 + saved // PHASES) + phase  # an index > 0 with this phase
        g = torch.cuda.CUDAGraph()
        self.cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=self.cap):
            for _ in range(length):
                self.step_fn(self.state.t)
        torch.cuda.synchronize()
        self.state.t = saved
        return g

    def segments(self, pos, K):
        out = []
        while K > 0:
            n = min(self.max_len, K)
            out.append((pos % PHASES, n))
            pos += n
            K -= n
        return out

    def prepare(self, K, blocks=PHASES):
        """Capture every graph that `blocks` consecutive blocks of K steps use (the schedule
        repeats after 4 blocks)."""
        pos = self.pos
        for _ in range(blocks):
            for key in self.segments(pos, K):
                if key not in self.graphs:
                    self.graphs[key] = self.capture(*key)
            pos += K

    def run(self, K):
        for key in self.segments(self.pos, K):
            self.graphs[key].replay()
        self.pos += K


def timed_blocks(torch, replayer, K, world, stream, before, min_ms=MIN_TIMED_MS, max_blocks=20000):
    """Time blocks of exactly K steps (device events, synchronised and barriered on both
    sides) until about min_ms of device time is covered; before() runs (on the host, GPU
    idle) after two untimed blocks that size the run.  Returns the per-block times (max
    over ranks), in ms."""
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def block():
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        replayer.run(K)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)

    probe = [block() for _ in range(2)]  # untimed: sizes the run
    n = max(3, min(max_blocks, int(min_ms / max(1e-3, min(probe))) + 1))
    n = int(max_over_ranks(n, world))
    before()
    torch.cuda.synchronize()
    times = [block() for _ in range(n)]
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor(times, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        times = t.tolist()
    return times


def block_summary(times, K):
    per_step = sorted(t / K for t in times)
    q = lambda f: per_step[min(len(per_step) - 1, int(f * (len(per_step) - 1) + 0.5))]
    return {"ms_per_step": statistics.median(per_step), "p10": q(0.1), "p90": q(0.9),
            "mean": sum(per_step) / len(per_step), "blocks": len(per_step), "timed_ms": sum(times)}


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------
def source_code_hash(path):
    """Hash of a source file's code: comments (//...) and blank lines do not count, so that a
    change of wording alone does not invalidate the counters."""
    import hashlib
    import re
    lines = []
    for line in open(path, encoding="utf-8").read().splitlines():
        code = re.sub(r"//.*$", "", line).rstrip()
        if code:
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def sources_code_hash(sources):
    """source_code_hash of one file, or of several (a list) taken together."""
    if isinstance(sources, str):
        return source_code_hash(os.path.join(ROOT, sources))
    import hashlib
    parts = ",".join(source_code_hash(os.path.join(ROOT, s)) for s in sources)
    return hashlib.sha256(parts.encode()).hexdigest()[:16]


def traffic_record(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's source code is
    unchanged since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path)).get(kernel)
        if not rec:
            return None
        h = sources_code_hash(rec["source"])
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("source_sha256_16") != h:
        return None
    return rec.get("dram_bytes_per_launch")


CHUNK_BYTES = 4096


def step_bytes(steps, B, N, V, esz, mode, recovery, tests, accepts):
    """Bytes the step algorithm must read over `steps` steps of B sequences, from the step's
    counters: every logit row a sequence's decisions need, once (a sequence with pending
    tokens: its N-1 anchor rows; one that then keeps all of them, or had none: rows
    N-1..2N-2; one that rejects, in the sampling mode: the residual's two rows, the anchor
    row K again and the previous call's MASK row N+K), plus the one chunk each draw reads
    again (4 KB; for the residual half a chunk of each row; argmax draws read none in the
    greedy mode).  A sequence rejects once per failed test: tests - accepts of them."""
    row = V * esz
    pending = steps * B - recovery
    rejecting = tests - accepts
    proposing = steps * B - rejecting            # all kept, or no pending tokens
    rows = pending * (N - 1) + proposing * N
    if mode == 0:
        rows += 2 * rejecting
    draws = 0 if mode == 1 else proposing * N + rejecting
    return rows * row + draws * CHUNK_BYTES


def stats_pass_bytes(steps, B, N, V, esz, recovery):
    """Bytes the statistics pass reads over `steps` steps: rows N-1..2N-2 of every sequence
    and the N-1 anchor rows of every sequence with pending tokens, each once (it runs before
    the decisions, so it reads the draw rows of sequences that will reject too)."""
    pending = steps * B - recovery
    return (steps * B * N + pending * (N - 1)) * V * esz


def run_ours(args, wl, rank, world, local_rank, fused=False, steps=None, min_ms=MIN_TIMED_MS, e2e=None,
             clocks=None):
    """The step on resident logits through isd_step (or isd_step_fused if fused), timed in
    graph-replayed blocks of `steps` steps."""
    import torch
    from diffusion_lm_decoding_isd_b300 import isd
    from diffusion_lm_decoding_isd_b300.synthetic import rotating_pool

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B, N, V = wl["B"], wl["N"], wl["V"]
    R = 2 * N - 1
    T, greedy = wl["temperature"], wl["greedy"]
    seed = 1234 + rank
    esz = 2 if wl["dtype"] == "bf16" else 4

    host = rotating_pool(B, N, V, wl["sigma_l"], wl["sigma_n"], seed, N_BUFFERS, wl["dtype"])
    tdt = torch.bfloat16 if wl["dtype"] == "bf16" else torch.float32
    pinned = []
    bufs = []
    for h in host:
        src = torch.from_numpy(h.view(np.int16) if wl["dtype"] == "bf16" else h)
        p = src.pin_memory()
        pinned.append(p.view(tdt))
        bufs.append(p.to(dev, non_blocking=False).view(tdt))
    torch.cuda.synchronize()

    state = isd.StepState(B, N, V, isd.ISD_BF16 if wl["dtype"] == "bf16" else isd.ISD_F32, dev, fused=fused)

    def step_fn(t):
        prev = bufs[(t - 1) % N_BUFFERS] if t > 0 else None
        state.step(bufs[t % N_BUFFERS], prev, T, greedy, seed)

    # eager warm-up
    W = max(args.warmup, 3)
    for t in range(W):
        step_fn(t)
    launches_per_step = isd.last_launch_count()
    torch.cuda.synchronize()

    K = args.steps if steps is None else steps
    rep = Replayer(torch, state, step_fn, dev)
    rep.prepare(K)
    # a graph of 8 steps with CUDA events around each kernel launch (which also serialises
    # the kernels) gives the per-kernel durations for the roofline
    isd.isd_profile_begin(8 * 4)
    g_prof = rep.capture(0, 8)
    stream = torch.cuda.current_stream()
    for _ in range(2):  # graph warm-up
        rep.run(K)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank) if (args.clocks if clocks is None else clocks) else None
    if sampler:
        sampler.start()
    times = timed_blocks(torch, rep, K, world, stream, before=state.diag.zero_, min_ms=min_ms)
    clock_rows = sampler.stop() if sampler else None
    diag = state.diag.cpu().numpy().astype(np.int64)
    summ = block_summary(times, K)
    n_steps = summ["blocks"] * K  # steps this rank ran in the timed blocks

    # per-kernel durations: replay the profiled graph (events re-recorded each replay)
    sums = {}
    for _ in range(32):
        g_prof.replay()
        for kind, name in isd.KERNEL_NAMES.items():
            ms, n = isd.isd_profile_read(kind)
            if n:
                a = sums.setdefault(name, [0.0, 0])
                a[0] += ms
                a[1] += n
    kern = {name: ms / n for name, (ms, n) in sums.items()}
    isd.isd_profile_end()
    torch.cuda.synchronize()

    emitted = int(diag[isd.DIAG_EMITTED])
    recovery = int(diag[isd.DIAG_RECOVERY])
    residuals = int(diag[isd.DIAG_RESIDUALS])
    tests = int(diag[isd.DIAG_TESTS])
    accepts = int(diag[isd.DIAG_ACCEPTS])
    assert diag[isd.DIAG_STATUS] == 0, "device status %d" % diag[isd.DIAG_STATUS]

    total_emitted = sum_over_ranks(emitted, world)
    ms_per_step = summ["ms_per_step"]
    tokens_per_step = total_emitted / n_steps  # all ranks
    value = tokens_per_step / (ms_per_step * 1e-3)

    nominal_bytes_step = B * R * V * esz
    alg_bytes = step_bytes(n_steps, B, N, V, esz, int(greedy), recovery, tests, accepts)
    hbm_peak, peak_kind = load_peaks()
    alg_bytes_launch = alg_bytes / n_steps
    if fused:
        # one kernel runs the whole step: its bytes are the step's
        dom = "isd_fused_step_kernel"
        dom_bytes_launch = alg_bytes_launch
    else:
        # the dominant kernel: the statistics pass, an HBM-bound scan
        dom = "isd_stats_kernel"
        dom_bytes_launch = stats_pass_bytes(n_steps, B, N, V, esz, recovery) / n_steps
    dom_ms = kern.get(dom)
    achieved = dom_bytes_launch / (dom_ms * 1e-3) / 1e9 if dom_ms else None
    traffic = traffic_record(dom)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": args.workload, "B": B, "N": N, "V": V, "logits_dtype": wl["dtype"],
            "temperature": T, "mode": MODE_NAMES[int(greedy)],
            "sigma_l": wl["sigma_l"], "sigma_n": wl["sigma_n"],
            "l2": "%d rotating logits buffers of %.1f MB each (> 126 MB L2)" % (N_BUFFERS, nominal_bytes_step / 1e6),
            "graph_steps": min(K, MAX_GRAPH_STEPS), "parallelism": "replicas" if world > 1 else "single",
            "entry": "isd_step_fused" if fused else "isd_step",
        },
        "timing": {"blocks": summ["blocks"], "steps_per_block": K, "timed_ms": round(summ["timed_ms"], 3),
                   "ms_per_step_p10": round(summ["p10"], 6), "ms_per_step_p90": round(summ["p90"], 6),
                   "ms_per_step_mean": round(summ["mean"], 6)},
        "logits_gbs": round(nominal_bytes_step * world / (ms_per_step * 1e-3) / 1e9, 1),
        "logits_frac_of_measured_hbm": round(nominal_bytes_step / (ms_per_step * 1e-3) / 1e9 / hbm_peak, 4),
        "logits_frac_of_nominal_8tbs": round(nominal_bytes_step / (ms_per_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "algorithmic_gbs": round(alg_bytes_launch / (ms_per_step * 1e-3) / 1e9, 1),
        "algorithmic_bytes_per_step": int(alg_bytes_launch),
        "tpf": round(emitted / (n_steps * B), 4),
        "accept_rate": round(accepts / max(1, tests), 4),
        **derived_tpf_metrics(emitted / (n_steps * B), N),
        "kernel_ms": {k: round(v, 5) for k, v in kern.items()},
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1) if achieved else None,
            "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4) if achieved else None,
            "traffic": traffic, "kernel": dom,
            "algorithmic_bytes_per_launch": int(dom_bytes_launch),
        },
        "gpu_launches": launches_per_step * n_steps,
    }
    if clock_rows is not None:
        out["clocks"] = summarize_clocks(clock_rows)

    # end to end through the public API with host buffers
    if args.e2e if e2e is None else e2e:
        out["e2e"] = run_e2e(args, wl, state, pinned, dev, seed, T, greedy, world)

    return out, host


def run_from_hidden(args, wl, rank, world, local_rank, workload=None, steps=None, min_ms=MIN_TIMED_MS, e2e=None):
    """isd_step_from_hidden: the tensor-core LM-head projection of the forward's hidden
    states, then the step on its logits.  The 1.245 GB weight is far larger than L2."""
    workload = workload or args.workload
    e2e = args.e2e if e2e is None else e2e
    import torch
    from diffusion_lm_decoding_isd_b300 import isd
    from diffusion_lm_decoding_isd_b300.synthetic import lm_head_inputs, rotating_pool

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B, N, V, K = wl["B"], wl["N"], wl["V"], wl["K"]
    R = 2 * N - 1
    M = B * R
    T, greedy = wl["temperature"], wl["greedy"]
    seed = 1234 + rank

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory().to(dev).view(torch.bfloat16)

    _, w_bits = lm_head_inputs(1, K, V, seed, sigma_w=wl["sigma_w"])
    weight = to_dev(w_bits)
    del w_bits
    host = rotating_pool(B, N, K, wl["sigma_l"], wl["sigma_n"], seed, N_BUFFERS, "bf16")
    pinned = [torch.from_numpy(h.view(np.int16)).pin_memory().view(torch.bfloat16) for h in host]
    hid = [p.to(dev) for p in pinned]
    logits = [torch.empty((B, R, V), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    torch.cuda.synchronize()
    state = isd.StepState(B, N, V, isd.ISD_BF16, dev, from_hidden=True)

    def step_fn(t):
        prev = logits[(t - 1) & 1] if t > 0 else None
        state.step_from_hidden(hid[t % N_BUFFERS], weight, logits[t & 1], prev, T, greedy, seed)

    W = max(args.warmup, 3)
    for t in range(W):
        step_fn(t)
    launches_per_step = isd.lm_head_last_launch_count() + isd.last_launch_count()
    torch.cuda.synchronize()
    Ks = steps if steps is not None else args.steps
    rep = Replayer(torch, state, step_fn, dev, max_len=8)
    rep.prepare(Ks)
    isd.isd_profile_begin(8 * 4)
    g_prof = rep.capture(0, 8)
    for _ in range(2):
        rep.run(Ks)
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if args.clocks else None
    if sampler:
        sampler.start()
    stream = torch.cuda.current_stream()
    times = timed_blocks(torch, rep, Ks, world, stream, before=state.diag.zero_, min_ms=min_ms)
    clock_rows = sampler.stop() if sampler else None
    summ = block_summary(times, Ks)
    n_steps = summ["blocks"] * Ks
    diag = state.diag.cpu().numpy().astype(np.int64)
    assert diag[isd.DIAG_STATUS] == 0, "device status %d" % diag[isd.DIAG_STATUS]
    sums = {}
    for _ in range(8):
        g_prof.replay()
        for kind, name in isd.KERNEL_NAMES.items():
            ms, n = isd.isd_profile_read(kind)
            if n:
                a = sums.setdefault(name, [0.0, 0])
                a[0] += ms
                a[1] += n
    kern = {name: ms / n for name, (ms, n) in sums.items()}
    isd.isd_profile_end()
    torch.cuda.synchronize()

    emitted = int(diag[isd.DIAG_EMITTED])
    total_emitted = sum_over_ranks(emitted, world)
    ms_per_step = summ["ms_per_step"]
    flops = 2.0 * M * K * V
    gemm_ms = kern.get("isd_lm_head_kernel")
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    burst = float(peaks.get("bf16_tflops", 1800.0))
    sustained = float(peaks.get("bf16_tflops_sustained", 1400.0))
    kind = "measured" if peaks else "fallback"
    achieved = flops / (gemm_ms * 1e-3) / 1e12 if gemm_ms else None
    out = {
        "metric": "verified tokens/s from hidden states (LM-head projection + ISD step), B=64 N=4 "
                  "V=151936 K=4096, 1 B300",
        "value": round(total_emitted / n_steps / (ms_per_step * 1e-3), 1), "unit": UNIT, "n_gpus": world,
        "steps": Ks, "warmup": W, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, "B": B, "N": N, "V": V, "K": K, "M": M,
                   "temperature": T, "mode": MODE_NAMES[int(greedy)],
                   "hidden": "N(0,1); clean rows = previous MASK rows + N(0,%.2f^2)" % wl["sigma_n"],
                   "weight": "N(0,%.2f^2), %.3f GB (> 126 MB L2)" % (wl["sigma_w"], V * K * 2 / 1e9),
                   "graph_steps": min(Ks, 8), "parallelism": "replicas" if world > 1 else "single"},
        "timing": {"blocks": summ["blocks"], "steps_per_block": Ks, "timed_ms": round(summ["timed_ms"], 3),
                   "ms_per_step_p10": round(summ["p10"], 6), "ms_per_step_p90": round(summ["p90"], 6),
                   "ms_per_step_mean": round(summ["mean"], 6)},
        "tpf": round(emitted / (n_steps * B), 4),
        **derived_tpf_metrics(emitted / (n_steps * B), N),
        "kernel_ms": {k: round(v, 5) for k, v in kern.items()},
        "weight_gbs": round(V * K * 2 / (gemm_ms * 1e-3) / 1e9, 1) if gemm_ms else None,
        "roofline": {
            "bound": "tensor", "achieved": round(achieved, 1) if achieved else None,
            "peak": sustained, "peak_kind": kind + " sustained bf16 (the kernel runs back to back for the "
                                                  "whole timed region)",
            "unit": "TFLOP/s", "frac": round(achieved / sustained, 4) if achieved else None,
            "burst_peak": burst, "frac_of_burst_peak": round(achieved / burst, 4) if achieved else None,
            "traffic": traffic_record("isd_lm_head_kernel"), "kernel": "isd_lm_head_kernel",
            "algorithmic_flops_per_launch": flops, "weight_bytes_per_launch": V * K * 2,
        },
        "gpu_launches": launches_per_step * n_steps,
    }
    if clock_rows is not None:
        out["clocks"] = summarize_clocks(clock_rows)
    if e2e:
        st = isd.StepState(B, N, V, isd.ISD_BF16, dev, from_hidden=True)
        stage = [torch.empty((B, R, K), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        out_acc = torch.empty(B, dtype=torch.int32).pin_memory()
        out_tok = torch.empty((B, R), dtype=torch.int32).pin_memory()
        steps = max(8, args.e2e_steps)
        total = 0
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for t in range(steps):
            stage[t & 1].copy_(pinned[t % N_BUFFERS], non_blocking=True)
            acc, tok, _ = st.step_from_hidden(stage[t & 1], weight, logits[t & 1],
                                              logits[(t - 1) & 1] if t > 0 else None, T, greedy, seed)
            out_acc.copy_(acc, non_blocking=True)
            out_tok.copy_(tok, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            total += int(out_acc.sum())
        el = max_over_ranks(time.perf_counter() - t0, world)
        out["e2e"] = {"value": round(sum_over_ranks(total, world) / el, 1), "unit": UNIT, "steps": steps,
                      "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": B * 4 + B * R * 4}
    return out, (host, seed)


def cpu_baseline_from_hidden(host_seed, wl, budget_s=15.0):
    """The oracle chain for one sequence: fp64 projection of its 2N-1 rows (weight in blocks of
    rows), rounding to bf16, then the fp64 step; consecutive steps until the budget is spent."""
    import oracle
    from oracle import lm_head as olm
    from diffusion_lm_decoding_isd_b300.synthetic import lm_head_inputs
    host, seed = host_seed
    B, N, V, K = wl["B"], wl["N"], wl["V"], wl["K"]
    R = 2 * N - 1
    _, w_bits = lm_head_inputs(1, K, V, seed, sigma_w=wl["sigma_w"])
    pend = -np.ones((1, N - 1), dtype=np.int32)
    pq = np.zeros((1, N - 1), dtype=np.float32)
    prev = None
    tokens = steps = 0
    t0 = time.perf_counter()
    while steps < 64 and (steps == 0 or time.perf_counter() - t0 < budget_s):
        h = host[steps % len(host)][0]  # sequence 0: [R][K]
        lg = np.empty((R, V), dtype=np.uint16)
        for v0 in range(0, V, 16384):
            lg[:, v0:v0 + 16384] = olm.f64_to_bf16_bits(olm.lm_head(h, w_bits[v0:v0 + 16384]))
        lg = lg.reshape(1, R, V)
        res = oracle.isd_step(lg, prev, pend, pq, N, wl["temperature"], wl["greedy"], seed, steps, dtype="bf16")
        tokens += int(res["accepted_len"].sum())
        pend = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)
        prev = lg
        steps += 1
    secs = time.perf_counter() - t0
    return {"value": round(tokens / secs, 2), "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": "sequence 0 of the batch, %d consecutive steps (fp64 numpy projection, which may use "
                      "every host core through BLAS, then the single-threaded fp64 C step), %.1f s"
                      % (steps, secs)}


MODE_NAMES = {0: "sampling", 1: "greedy", 2: "argmax proposals, sampled verification"}
R_ISD_OVERHEAD = 1.12  # cost of one R-ISD forward relative to a plain one


def derived_tpf_metrics(tpf, N):
    """Metrics the pages derive from tokens per forward: the compute efficiency TPF^2 over the
    queries per forward, 2N-1 (ai.arkapp.pw blog, section "為什麼 I-DLM 能在高並發下保持高效？";
    1.22 at N=4, p=0.9), and the lossless R-ISD speedup TPF / alpha with the gated adapter's
    overhead alpha = 1.12 (de.news.hada.io summary, section "Speedup Factor Explorer")."""
    return {"compute_efficiency": round(tpf * tpf / (2 * N - 1), 4),
            "r_isd_speedup": round(tpf / R_ISD_OVERHEAD, 4)}


SWEEP_N = (2, 3, 4, 8)
SWEEP_SIGMA_N = (0.1, 0.5, 1.0, 2.0)


def tpf_closed_form(p, N):
    """Tokens per forward of ISD at constant per-token acceptance p:
    (2 + p + ... + p^(N-2)) / (2 - p^(N-1))."""
    return (2.0 + sum(p ** i for i in range(1, N - 1))) / (2.0 - p ** (N - 1))


def device_pool(B, N, V, sigma_l, sigma_n, seed, n_buffers, dev):
    """Like synthetic.rotating_pool, generated on the device with torch's seeded normal
    generator (inputs only): buffer k's clean rows 0..N-2 are buffer k-1's MASK rows plus
    N(0, sigma_n^2) noise, every other row N(0, sigma_l^2); bf16."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    R = 2 * N - 1
    bufs = [(torch.randn((B, R, V), generator=g, device=dev) * sigma_l).to(torch.bfloat16)
            for _ in range(n_buffers)]
    for k in range(n_buffers):
        noise = torch.randn((B, N - 1, V), generator=g, device=dev) * sigma_n
        bufs[k][:, :N - 1] = (bufs[k - 1][:, N:].float() + noise).to(torch.bfloat16)
    return bufs


def run_sweep(args, rank, local_rank, B=64, V=151936, sigma_l=3.0, T=1.0, steps=256, warm=8,
              Ns=SWEEP_N, sigmas=SWEEP_SIGMA_N):
    """Acceptance / stride sweep: for each (N, sigma_n) the measured tokens per forward, the
    measured per-token acceptance p_hat = accepts / tests, and the closed form at p_hat."""
    import torch
    from diffusion_lm_decoding_isd_b300 import isd
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    rows = []
    for N in Ns:
        for sn in sigmas:
            bufs = device_pool(B, N, V, sigma_l, sn, 4321 + 97 * N + int(sn * 100), 3, dev)
            st = isd.StepState(B, N, V, isd.ISD_BF16, dev)
            for t in range(warm):
                st.step(bufs[t % 3], bufs[(t - 1) % 3] if t else None, T, False, 99)
            st.diag.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for t in range(warm, warm + steps):
                st.step(bufs[t % 3], bufs[(t - 1) % 3], T, False, 99)
            e1.record()
            torch.cuda.synchronize()
            d = st.diag.cpu().numpy().astype(np.int64)
            assert d[isd.DIAG_STATUS] == 0, d
            p_hat = d[isd.DIAG_ACCEPTS] / max(1, d[isd.DIAG_TESTS])
            tpf = d[isd.DIAG_EMITTED] / (steps * B)
            cf = tpf_closed_form(p_hat, N)
            rows.append({"N": N, "sigma_n": sn, "p_hat": round(float(p_hat), 4), "tpf": round(float(tpf), 4),
                         "tpf_closed_form": round(cf, 4), "rel_diff": round(float(tpf / cf - 1.0), 4),
                         **derived_tpf_metrics(float(tpf), N),
                         "us_per_step": round(e0.elapsed_time(e1) * 1e3 / steps, 2),
                         "logits_gbs": round(B * (2 * N - 1) * V * 2 * steps / (e0.elapsed_time(e1) * 1e-3) / 1e9,
                                             1)})
            del bufs, st
            torch.cuda.empty_cache()
    return rows


def run_e2e(args, wl, state, pinned, dev, seed, T, greedy, world):
    """Every step: H2D of the step's logits from pinned host memory, isd_step,
    D2H of accepted_len and tokens_out, synchronize.  Uses a fresh state."""
    import torch
    from diffusion_lm_decoding_isd_b300 import isd
    B, N, V = wl["B"], wl["N"], wl["V"]
    R = 2 * N - 1
    tdt = pinned[0].dtype
    stage = [torch.empty((B, R, V), dtype=tdt, device=dev) for _ in range(2)]
    st = isd.StepState(B, N, V, isd.ISD_BF16 if tdt == torch.bfloat16 else isd.ISD_F32, dev)
    out_acc = torch.empty(B, dtype=torch.int32).pin_memory()
    out_tok = torch.empty((B, R), dtype=torch.int32).pin_memory()
    steps = max(8, args.e2e_steps)
    total = 0
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for t in range(steps):
        cur = stage[t & 1]
        cur.copy_(pinned[t % N_BUFFERS], non_blocking=True)
        acc, tok, _ = st.step(cur, stage[(t - 1) & 1] if t > 0 else None, T, greedy, seed)
        out_acc.copy_(acc, non_blocking=True)
        out_tok.copy_(tok, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        total += int(out_acc.sum())
    el = time.perf_counter() - t0
    barrier(world)
    el = max_over_ranks(el, world)
    total = sum_over_ranks(total, world)
    esz = pinned[0].element_size()
    return {"value": round(total / el, 1), "unit": UNIT, "steps": steps,
            "h2d_bytes_per_step": B * R * V * esz, "d2h_bytes_per_step": B * 4 + B * R * 4}


# ------------------------------------------------------------------------------------
# the oracle on the host cores
# ------------------------------------------------------------------------------------
def oracle_chain(host_bufs, wl, seqs, max_steps, budget_s, steps_exact=None, pool=None):
    """Run the fp64 oracle over consecutive pool buffers for the given sequences, carrying
    its own pending state; single-threaded, or over the host cores through `pool` (an
    oracle.parallel.OraclePool).  Returns (tokens, seconds, steps)."""
    import oracle
    B, N, V = wl["B"], wl["N"], wl["V"]
    T, greedy = wl["temperature"], wl["greedy"]
    nb = len(host_bufs)
    sub = [np.ascontiguousarray(h[seqs]) for h in host_bufs]
    pend = -np.ones((len(seqs), N - 1), dtype=np.int32)
    pq = np.zeros((len(seqs), N - 1), dtype=np.float32)
    step = pool.isd_step if pool is not None else oracle.isd_step
    tokens = 0
    t0 = time.perf_counter()
    steps = 0
    while True:
        if steps_exact is not None and steps >= steps_exact:
            break
        if steps_exact is None and steps >= 1 and (steps >= max_steps or time.perf_counter() - t0 > budget_s):
            break
        prev = sub[(steps - 1) % nb] if steps > 0 else None
        res = step(sub[steps % nb], prev, pend, pq, N, T, greedy, 1234, steps, dtype=wl["dtype"])
        tokens += int(res["accepted_len"].sum())
        pend = res["tokens_out"][:, N:].astype(np.int32)
        pq = res["new_q"].astype(np.float32)
        steps += 1
    return tokens, time.perf_counter() - t0, steps


def cpu_baseline(host_bufs, wl, budget_s=15.0):
    """The oracle on the host: the full batch over all host cores (one worker process per
    core, sequences split among them), and single-threaded; each for about half the budget."""
    from oracle.parallel import OraclePool, host_cores
    seqs = list(range(wl["B"]))
    with OraclePool() as pool:
        oracle_chain(host_bufs, wl, seqs, max_steps=1, budget_s=0, pool=pool)  # workers started
        tokens, secs, steps = oracle_chain(host_bufs, wl, seqs, max_steps=256, budget_s=budget_s / 2, pool=pool)
        workers = pool.workers
    t1, s1, n1 = oracle_chain(host_bufs, wl, seqs, max_steps=64, budget_s=budget_s / 2)
    return {"value": round(tokens / secs, 2), "unit": UNIT, "cores": workers, "kind": "oracle", "nproc": host_cores(),
            "sample": "%d consecutive steps of the full B=%d batch, fp64 C oracle in %d worker processes "
                      "(sequences split among them), %.1f s" % (steps, wl["B"], workers, secs),
            "single_thread": {"value": round(t1 / s1, 2), "unit": UNIT, "cores": 1,
                              "sample": "%d consecutive steps of the full batch, %.1f s" % (n1, s1)}}


REFERENCE_BUDGET_S = 120.0


def run_reference(args, wl, rank, world):
    if rank != 0:
        return None
    if wl.get("kind") == "from_hidden":
        from diffusion_lm_decoding_isd_b300.synthetic import rotating_pool
        host = rotating_pool(wl["B"], wl["N"], wl["K"], wl["sigma_l"], wl["sigma_n"], 1234, N_BUFFERS, "bf16")
        cb = cpu_baseline_from_hidden((host, 1234), wl, args.cpu_budget)
        return {
            "metric": "verified tokens/s from hidden states (LM-head projection + ISD step), B=64 N=4 "
                      "V=151936 K=4096, 1 B300",
            "value": cb["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "B": wl["B"], "N": wl["N"], "V": wl["V"], "K": wl["K"],
                       "reference": "fp64 CPU oracle (oracle/lm_head.py + oracle/isd_oracle.c); one sequence"},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    from oracle.parallel import OraclePool
    from diffusion_lm_decoding_isd_b300.synthetic import rotating_pool
    host = rotating_pool(wl["B"], wl["N"], wl["V"], wl["sigma_l"], wl["sigma_n"], 1234,
                         N_BUFFERS, wl["dtype"])
    W = max(args.warmup, 3)
    K = args.steps
    B = wl["B"]
    with OraclePool() as pool:
        # one full-batch step sizes the per-step sample so that the K steps end within the budget
        _, t_full, _ = oracle_chain(host, wl, list(range(B)), 0, 0, steps_exact=1, pool=pool)
        nseq = B if K * t_full <= REFERENCE_BUDGET_S else max(1, int(B * REFERENCE_BUDGET_S / (K * t_full)))
        use_pool = pool if nseq >= pool.workers else None
        cores = pool.workers if use_pool else 1
        seqs = list(range(nseq))
        oracle_chain(host, wl, seqs, 0, 0, steps_exact=min(W, 3), pool=use_pool)
        tokens, secs, steps = oracle_chain(host, wl, seqs, 0, 0, steps_exact=K, pool=use_pool)
    value = tokens / secs
    sample = ("%s of the B=%d batch per step, %d consecutive steps, fp64 C oracle %s"
              % ("all %d sequences" % B if nseq == B else "the first %d sequences" % nseq, B, K,
                 "in %d worker processes" % cores if cores > 1 else "single-threaded"))
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(secs * 1e3 / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": args.workload, "B": wl["B"], "N": wl["N"], "V": wl["V"],
                   "logits_dtype": wl["dtype"], "temperature": wl["temperature"],
                   "mode": MODE_NAMES[int(wl["greedy"])],
                   "reference": "fp64 CPU oracle (oracle/isd_oracle.c)"},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def parse_args(argv=None):
    from diffusion_lm_decoding_isd_b300.synthetic import WORKLOADS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-clocks", dest="clocks", action="store_false")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--sweep", action="store_true",
                    help="acceptance/stride sweep over N and the anchor noise; one JSON line per point")
    ap.add_argument("--sweep-steps", type=int, default=256)
    ap.add_argument("--no-from-hidden", dest="from_hidden", action="store_false",
                    help="leave the from-hidden workload out of the default workload's line")
    ap.add_argument("--fused", action="store_true",
                    help="time isd_step_fused (the step as one persistent kernel) instead of isd_step")
    ap.add_argument("--no-fused-line", dest="fused_line", action="store_false",
                    help="leave the isd_step_fused timing out of the default workload's line")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    from diffusion_lm_decoding_isd_b300.synthetic import WORKLOADS
    wl = dict(WORKLOADS[args.workload])
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.sweep:
        if rank == 0:
            rows = run_sweep(args, rank, local_rank, steps=args.sweep_steps)
            for r in rows:
                print(json.dumps(dict(sweep="acceptance/stride, B=64 V=151936 bf16 sigma_l=3 T=1", **r)),
                      flush=True)
        return
    if args.impl == "reference":
        out = run_reference(args, wl, rank, world)
    elif wl.get("kind") == "from_hidden":
        out, host_seed = run_from_hidden(args, wl, rank, world, local_rank)
        if rank == 0 and world == 1 and args.cpu_baseline:
            out["cpu_baseline"] = cpu_baseline_from_hidden(host_seed, wl, args.cpu_budget)
    else:
        out, host = run_ours(args, wl, rank, world, local_rank, fused=args.fused)
        if args.fused_line and not args.fused and args.workload == DEFAULT_WORKLOAD:
            # the same step as one persistent kernel (isd_step_fused), timed in the same run
            fu, _ = run_ours(args, wl, rank, world, local_rank, fused=True, steps=min(args.steps, FUSED_STEPS),
                             min_ms=300.0, e2e=False, clocks=False)
            out["fused_step"] = {k: fu[k] for k in ("metric", "value", "unit", "steps", "ms_per_step", "timing",
                                                    "tpf", "kernel_ms", "roofline", "gpu_launches") if k in fu}
            out["fused_step"]["entry"] = "isd_step_fused"
        if args.from_hidden and args.workload == DEFAULT_WORKLOAD:
            # the tensor-core path, timed in the same run: nested in the same line
            fh_name = "from_hidden_b64_n4_k4096"
            fh, _ = run_from_hidden(args, dict(WORKLOADS[fh_name]), rank, world, local_rank, workload=fh_name,
                                    steps=FROM_HIDDEN_STEPS, min_ms=300.0, e2e=False)
            out["from_hidden"] = {k: fh[k] for k in ("metric", "value", "unit", "steps", "ms_per_step", "config",
                                                     "timing", "tpf", "kernel_ms", "weight_gbs", "roofline",
                                                     "gpu_launches", "clocks") if k in fh}
        if rank == 0 and world == 1 and args.cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(host, wl, args.cpu_budget)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
