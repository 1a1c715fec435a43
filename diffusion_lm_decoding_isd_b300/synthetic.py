"""Seeded synthetic forward logits for the ISD step.

This module generates inputs only.  It holds none of the decoding method's
arithmetic, so both the CUDA path and the CPU oracle can be fed the same
bytes.  The model-free stand-in follows the shape of one ISD forward: per
sequence 2N-1 rows over the vocabulary, where row i-1 (the clean row that
verifies pending token x_i) is the previous forward's MASK row N-1+i (which
proposed x_i) plus Gaussian noise, so the anchor and proposal distributions
differ by a controlled amount; the anchor row N-1 and the MASK rows are fresh.
"""
import numpy as np


def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (nearest, ties to even); uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b):
    """bf16 bit patterns (uint16) -> float32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _encode(x, dtype):
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError("dtype must be 'bf16' or 'f32'")


def _decode(x, dtype):
    return bf16_bits_to_f32(x) if dtype == "bf16" else np.asarray(x, dtype=np.float32)


class ForwardStream:
    """Successive forwards [B][2N-1][V] of a stationary batch.

    Fresh rows ~ N(0, sigma_l^2).  For t > 0, clean row i-1 (i = 1..N-1) of
    forward t equals MASK row N-1+i of forward t-1 plus N(0, sigma_n^2) noise.
    Values are rounded to the storage dtype ("bf16" as uint16 bit patterns, or
    "f32").
    """

    def __init__(self, B, N, V, sigma_l, sigma_n, seed, dtype="bf16"):
        self.B, self.N, self.V = B, N, V
        self.sigma_l, self.sigma_n, self.dtype = float(sigma_l), float(sigma_n), dtype
        self.rng = np.random.default_rng(seed)
        self.prev = None

    def next(self):
        B, N, V = self.B, self.N, self.V
        R = 2 * N - 1
        x = self.rng.standard_normal((B, R, V), dtype=np.float32)
        x *= np.float32(self.sigma_l)
        if self.prev is not None:
            noise = self.rng.standard_normal((B, N - 1, V), dtype=np.float32)
            noise *= np.float32(self.sigma_n)
            x[:, :N - 1] = _decode(self.prev[:, N:], self.dtype) + noise
        out = _encode(x, self.dtype)
        self.prev = out
        return out


def rotating_pool(B, N, V, sigma_l, sigma_n, seed, n_buffers, dtype="bf16"):
    """n_buffers forwards that can be cycled forever: buffer k's clean rows
    0..N-2 are buffer (k-1) mod n_buffers's MASK rows plus noise."""
    rng = np.random.default_rng(seed)
    R = 2 * N - 1
    bufs = []
    for _ in range(n_buffers):
        x = rng.standard_normal((B, R, V), dtype=np.float32)
        x *= np.float32(sigma_l)
        bufs.append(x)
    for k in range(n_buffers):
        prev_mask = _decode(_encode(bufs[k - 1][:, N:], dtype), dtype)
        noise = rng.standard_normal((B, N - 1, V), dtype=np.float32)
        noise *= np.float32(sigma_n)
        bufs[k][:, :N - 1] = prev_mask + noise
    return [_encode(x, dtype) for x in bufs]


# The workloads the step is measured and checked on (shape, value recipe).
WORKLOADS = {
    "tiny_f32": dict(B=1, N=2, V=256, sigma_l=2.0, sigma_n=0.3, dtype="f32", temperature=1.0,
                     greedy=False, steps=64),
    "b8_n4_v151936": dict(B=8, N=4, V=151936, sigma_l=3.0, sigma_n=0.5, dtype="bf16",
                          temperature=1.0, greedy=False, steps=256),
    "b64_n4_v151936_greedy": dict(B=64, N=4, V=151936, sigma_l=3.0, sigma_n=0.5, dtype="bf16",
                                  temperature=1.0, greedy=True, steps=512),
    "b64_n4_v151936_t0.7": dict(B=64, N=4, V=151936, sigma_l=3.0, sigma_n=0.5, dtype="bf16",
                                temperature=0.7, greedy=False, steps=512),
    # argmax proposals (q = 1) verified by sampling (the step's greedy argument = 2)
    "b64_n4_v151936_argmax_propose": dict(B=64, N=4, V=151936, sigma_l=3.0, sigma_n=0.5, dtype="bf16",
                                          temperature=1.0, greedy=2, steps=512),
    # hidden states [64*7, 4096] ~ N(0, 1) whose clean rows are the previous forward's MASK
    # rows plus N(0, 0.39^2) (about N(0, 0.5^2) on the logits through the weight below), and
    # an LM-head weight [151936, 4096] ~ N(0, 0.02^2)
    "from_hidden_b64_n4_k4096": dict(kind="from_hidden", B=64, N=4, V=151936, K=4096, sigma_l=1.0,
                                     sigma_n=0.39, sigma_w=0.02, dtype="bf16", temperature=1.0,
                                     greedy=False, steps=64),
    "from_hidden_b64_n4_k4096_greedy": dict(kind="from_hidden", B=64, N=4, V=151936, K=4096, sigma_l=1.0,
                                            sigma_n=0.39, sigma_w=0.02, dtype="bf16", temperature=1.0,
                                            greedy=True, steps=64),
}


def lm_head_inputs(M, K, V, seed, sigma_h=1.0, sigma_w=0.02, grid=False, block=16384, w_den=256):
    """Seeded inputs of the LM-head projection as bf16 bit patterns (uint16):
    hidden [M][K] ~ N(0, sigma_h^2) and weight [V][K] ~ N(0, sigma_w^2), or with
    grid=True hidden in {-8..8}/8 and weight in {-8..8}/w_den (a power of two >= 8;
    every fp32 partial sum of such products is exact for K <= 2^14).  On the grid
    the logits have standard deviation about 0.375 * sqrt(K) * 8 / w_den.  The
    weight is generated in blocks of `block` rows, block j from seed (seed, 1, j),
    so that any rows can be regenerated alone (weight_rows)."""
    rng = np.random.default_rng([seed, 0])
    if grid:
        h = rng.integers(-8, 9, size=(M, K)).astype(np.float32) / 8.0
    else:
        h = rng.standard_normal((M, K), dtype=np.float32) * np.float32(sigma_h)
    hidden = f32_to_bf16_bits(h)
    weight = np.empty((V, K), dtype=np.uint16)
    for j, r0 in enumerate(range(0, V, block)):
        weight[r0:r0 + block] = _weight_block(j, min(block, V - r0), K, seed, sigma_w, grid, w_den)
    return hidden, weight


def _weight_block(j, rows, K, seed, sigma_w, grid, w_den=256):
    rng = np.random.default_rng([seed, 1, j])
    if grid:
        w = rng.integers(-8, 9, size=(rows, K)).astype(np.float32) / float(w_den)
    else:
        w = rng.standard_normal((rows, K), dtype=np.float32) * np.float32(sigma_w)
    return f32_to_bf16_bits(w)


def weight_rows(rows, K, V, seed, sigma_w=0.02, grid=False, block=16384):
    """Rows `rows` of the weight lm_head_inputs(..., seed, ...) generates."""
    rows = np.asarray(rows)
    out = np.empty((len(rows), K), dtype=np.uint16)
    for j in np.unique(rows // block):
        r0 = int(j) * block
        blk = _weight_block(int(j), min(block, V - r0), K, seed, sigma_w, grid)
        sel = np.nonzero(rows // block == j)[0]
        out[sel] = blk[rows[sel] - r0]
    return out


def grid_hidden_stream(B, N, K, steps, seed, flip=0.1):
    """Successive forwards' hidden states [B][2N-1][K] on the grid {-8..8}/8 (bf16 bit
    patterns): fresh rows uniform on the grid; from the second forward on, clean row i-1 is
    the previous forward's MASK row N-1+i with a fraction `flip` of its entries moved by one
    grid step (clipped), so that proposals are often accepted."""
    rng = np.random.default_rng([seed, 2])
    R = 2 * N - 1
    out, prev = [], None
    for _ in range(steps):
        h = rng.integers(-8, 9, size=(B, R, K))
        if prev is not None:
            step = rng.integers(-1, 2, size=(B, N - 1, K)) * (rng.random((B, N - 1, K)) < flip)
            h[:, :N - 1] = np.clip(prev[:, N:] + step, -8, 8)
        prev = h
        out.append(f32_to_bf16_bits(h.astype(np.float32) / 8.0))
    return out
