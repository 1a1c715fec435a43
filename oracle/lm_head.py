"""fp64 oracle of the LM-head projection (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this module; the product path never does.

What it computes ("Introspective Diffusion Language Models", ai.arkapp.pw
blog, section "I-DLM 如何解決這些問題": one forward scores every clean and MASK
position; its output layer maps each position's final hidden state to logits
over the vocabulary):

    logits[m][v] = round_bf16( sum_k hidden[m][k] * weight[v][k] )

with hidden [M][K] and weight [V][K] given as bf16 bit patterns (uint16).  The
sum is taken in fp64 (a library matmul; every product of two bf16 values is
exact in fp64, and for the sizes used here the fp64 sum is within 2^-40 of the
exact real sum relative to sum_k |h_k w_k|), then rounded once to the nearest
bf16 value, ties to even.  No intermediate rounding to fp32.

Parity of the GPU kernel (fp32 accumulation) is checked against ``exact``
together with ``abs_sum`` (sum_k |h_k w_k|), which bounds the accumulation
error.
"""
import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")      # largest finite bf16
BF16_MIN_NORMAL = 2.0 ** -126
BF16_SUBNORMAL_STEP = 2.0 ** -133           # spacing of bf16 subnormals


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) -> their exact values as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_bf16(x):
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float64.  bf16 keeps 8 significant bits and fp32's exponent range; values
    beyond the largest finite bf16 after rounding become +-inf."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    a = np.abs(x)
    sub = a < BF16_MIN_NORMAL
    # normal range: x = f * 2^e with 0.5 <= |f| < 1, keep 8 significant bits
    f, e = np.frexp(np.where(sub, 1.0, x))
    out[:] = np.ldexp(np.rint(f * 256.0), e - 8)
    # subnormal range: a fixed grid of 2^-133
    out[sub] = np.rint(x[sub] / BF16_SUBNORMAL_STEP) * BF16_SUBNORMAL_STEP
    over = np.abs(out) > BF16_MAX
    out[over] = np.copysign(np.inf, x[over])
    nan = np.isnan(x)
    out[nan] = np.nan
    return out


def f64_to_bf16_bits(x):
    """bf16 bit patterns of float64 values that are already bf16 values."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def exact(hidden_bits, weight_bits):
    """sum_k hidden[m][k] * weight[v][k] in fp64, [M][V]."""
    h = bf16_to_f64(hidden_bits)
    w = bf16_to_f64(weight_bits)
    return h @ w.T


def abs_sum(hidden_bits, weight_bits):
    """sum_k |hidden[m][k] * weight[v][k]| in fp64, [M][V]."""
    return np.abs(bf16_to_f64(hidden_bits)) @ np.abs(bf16_to_f64(weight_bits)).T


def lm_head(hidden_bits, weight_bits):
    """The projection's logits as bf16 values (float64 array), [M][V]."""
    return round_bf16(exact(hidden_bits, weight_bits))
