"""The oracle's step over groups of sequences in worker processes (test infrastructure).

Only ``tests/`` and ``bench.py``'s CPU legs use this module.  Sequences are
independent in the step, so a batch splits into contiguous groups of sequences,
each run by the plain single-threaded oracle in its own process; the uniforms of
sequence b are those of its place in the whole batch (Philox counter
(step, b, row)), passed explicitly.  The workers are started with the ``spawn``
method (never forked from a process that may hold a CUDA context).  Logits
reach the workers through memory-mapped files, written once per step.
"""
import multiprocessing as mp
import os
import tempfile

import numpy as np

_maps = {}  # worker side: path -> (mtime, memmap)


def _view(meta):
    if meta is None:
        return None
    path, shape, dtype = meta
    st = os.stat(path)
    key = (path, st.st_mtime_ns, st.st_size)
    m = _maps.get(path)
    if m is None or m[0] != key:
        m = (key, np.memmap(path, dtype=dtype, mode="r", shape=shape))
        _maps[path] = m
    return m[1]


def _run_group(args):
    import oracle
    (lmeta, pmeta, pend, pq, b0, b1, N, T, greedy, seed, step, dtype, near_tol) = args
    R = 2 * N - 1
    lg = np.ascontiguousarray(_view(lmeta)[b0:b1])
    pv = _view(pmeta)
    pv = None if pv is None else np.ascontiguousarray(pv[b0:b1])
    ua = np.zeros((b1 - b0, R))
    us = np.zeros((b1 - b0, R))
    for b in range(b0, b1):
        for r in range(R):
            ua[b - b0, r], us[b - b0, r] = oracle.row_uniforms(seed, step, b, r)
    return oracle.isd_step_u(lg, pv, pend, pq, N, T, greedy, ua, us, dtype=dtype, near_tol=near_tol)


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """oracle.isd_step over all host cores (or `workers` processes)."""

    def __init__(self, workers=None):
        self.workers = max(1, workers or host_cores())
        self.pool = mp.get_context("spawn").Pool(self.workers)
        # memory-backed files when the host has them (no disk traffic per step)
        shm = "/dev/shm"
        self.dir = tempfile.mkdtemp(prefix="isd_oracle_", dir=shm if os.path.isdir(shm) else None)

    def _put(self, key, arr):
        if arr is None:
            return None
        path = os.path.join(self.dir, key)
        # rewrite in place when the size is unchanged (no truncation under a worker's map)
        same = os.path.exists(path) and os.path.getsize(path) == arr.nbytes
        m = np.memmap(path, dtype=arr.dtype, mode="r+" if same else "w+", shape=arr.shape)
        m[...] = arr
        m.flush()
        del m
        return (path, arr.shape, arr.dtype.str)

    def isd_step(self, logits, prev_logits, pending_tokens, pending_q, N, temperature, greedy,
                 seed, step, dtype="bf16", near_tol=None):
        import oracle
        near_tol = oracle.NEAR_TOL if near_tol is None else near_tol
        enc = np.uint16 if dtype == "bf16" else np.float32
        lg = np.ascontiguousarray(logits, dtype=enc)
        B = lg.shape[0]
        pend = np.ascontiguousarray(np.asarray(pending_tokens, dtype=np.int32).reshape(B, N - 1))
        pq = np.ascontiguousarray(np.asarray(pending_q, dtype=np.float32).reshape(B, N - 1))
        lmeta = self._put("logits", lg)
        pmeta = self._put("prev", None if prev_logits is None else np.ascontiguousarray(prev_logits, dtype=enc))
        n = min(self.workers, B)
        edges = [B * i // n for i in range(n + 1)]
        jobs = [(lmeta, pmeta, pend[edges[i]:edges[i + 1]], pq[edges[i]:edges[i + 1]], edges[i], edges[i + 1],
                 N, float(temperature), int(greedy), int(seed), int(step), dtype, float(near_tol))
                for i in range(n) if edges[i + 1] > edges[i]]
        parts = self.pool.map(_run_group, jobs)
        return {k: np.concatenate([p[k] for p in parts], axis=0) for k in parts[0]}

    def close(self):
        self.pool.close()
        self.pool.join()
        for name in os.listdir(self.dir):
            os.unlink(os.path.join(self.dir, name))
        os.rmdir(self.dir)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
