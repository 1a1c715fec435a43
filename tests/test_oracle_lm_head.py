"""Pins of the fp64 LM-head oracle to facts outside itself: torch's fp32->bf16
conversion (round to nearest even) on values fp32 holds exactly, hand-worked
rounding cases where rounding through fp32 first would be wrong, brute force in
exact rational arithmetic, and one-hot / closed-form products that fix which
operand is transposed."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import lm_head as olm
from diffusion_lm_decoding_isd_b300.synthetic import lm_head_inputs, weight_rows, f32_to_bf16_bits


def _bits(values):
    return olm.f64_to_bf16_bits(np.asarray(values, dtype=np.float64))


def test_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(7)
    # random fp32 bit patterns over the whole finite range, plus exact ties
    u = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    ties = (rng.integers(0, 2**16, size=5000, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    t = ties.view(np.float32)
    x = np.concatenate([x, t[np.isfinite(t)]])
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = olm.round_bf16(x.astype(np.float64))
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), (x[~same][:5], got[~same][:5], want[~same][:5])


@pytest.mark.parametrize("x,want", [
    (1.0 + 2.0**-8, 1.0),                        # tie -> even (mantissa 0)
    (1.0 + 3 * 2.0**-8, 1.0 + 2.0**-6),          # tie -> even (mantissa 2)
    (1.0 + 2.0**-8 + 2.0**-30, 1.0 + 2.0**-7),   # just above the tie: fp32 first would give 1.0
    (-(1.0 + 2.0**-8 + 2.0**-30), -(1.0 + 2.0**-7)),
    (3.0 * 2.0**-140, 2.0**-133 * 0.0),          # below half a subnormal step -> 0
    (2.0**-133 * 0.5 + 2.0**-160, 2.0**-133),    # just above half a subnormal step
    (float.fromhex("0x1.ff8p127"), np.inf),      # rounds past the largest finite bf16
    (float.fromhex("0x1.fe7p127"), float.fromhex("0x1.fep127")),
    (0.0, 0.0),
])
def test_round_hand_cases(x, want):
    got = olm.round_bf16(np.array([x]))[0]
    assert got == want, (x, got, want)


def _brute(h, w):
    """Exact rational sums, each rounded to bf16 by counting ulps (Python's
    round() of a Fraction rounds halves to even)."""
    M, K = h.shape
    V = w.shape[0]
    out = np.zeros((M, V))
    for m in range(M):
        for v in range(V):
            s = sum((Fraction(float(h[m, k])) * Fraction(float(w[v, k])) for k in range(K)), Fraction(0))
            if s == 0:
                continue
            a = abs(s)
            e = 0
            while a >= 2:
                a /= 2
                e += 1
            while a < 1:
                a *= 2
                e -= 1
            ulp = Fraction(2) ** (e - 7)
            out[m, v] = float(round(s / ulp) * ulp)
    return out


@pytest.mark.parametrize("M,K,V", [(3, 5, 4), (2, 17, 7), (5, 8, 3)])
def test_lm_head_brute_force(M, K, V):
    rng = np.random.default_rng(M * 100 + K)
    h = f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    w = f32_to_bf16_bits(rng.standard_normal((V, K), dtype=np.float32) * np.float32(0.3))
    want = _brute(olm.bf16_to_f64(h), olm.bf16_to_f64(w))
    got = olm.lm_head(h, w)
    np.testing.assert_array_equal(got, want)


def test_lm_head_one_hot_selects_weight_columns():
    # hidden row m = e_{k_m}: logits[m][v] = weight[v][k_m], exactly
    K, V = 24, 11
    rng = np.random.default_rng(3)
    w = f32_to_bf16_bits(rng.standard_normal((V, K), dtype=np.float32))
    ks = [0, 5, 23, 7]
    h = np.zeros((len(ks), K))
    for m, k in enumerate(ks):
        h[m, k] = 1.0
    got = olm.lm_head(_bits(h), w)
    wf = olm.bf16_to_f64(w)
    for m, k in enumerate(ks):
        np.testing.assert_array_equal(got[m], wf[:, k])


def test_lm_head_closed_form_arange():
    # hidden row m = (m+1) * ones, weight row v = (v, v, ..., v) / 8 + arange(K) / 64
    # sum = (m+1) * (K v / 8 + K (K-1) / 128)
    M, K, V = 3, 16, 5
    h = np.repeat(np.arange(1, M + 1, dtype=np.float64)[:, None], K, axis=1)
    w = np.arange(V, dtype=np.float64)[:, None] / 8.0 + np.arange(K, dtype=np.float64)[None, :] / 64.0
    got = olm.exact(_bits(h), _bits(w))
    want = np.array([[(m + 1) * (K * v / 8.0 + K * (K - 1) / 128.0) for v in range(V)] for m in range(M)])
    np.testing.assert_array_equal(got, want)
    # a non-square product distinguishes weight from its transpose
    assert got.shape == (M, V)


def test_abs_sum_bounds_exact():
    h, w = lm_head_inputs(4, 64, 9, seed=5)
    e = olm.exact(h, w)
    a = olm.abs_sum(h, w)
    assert (np.abs(e) <= a + 1e-12).all()


def test_weight_rows_regenerates_blocks():
    _, w = lm_head_inputs(2, 16, 50, seed=9, block=16)
    rows = np.array([0, 15, 16, 49, 33])
    np.testing.assert_array_equal(weight_rows(rows, 16, 50, seed=9, block=16), w[rows])


def test_grid_inputs_are_bf16_exact_and_small():
    h, w = lm_head_inputs(8, 32, 20, seed=2, grid=True)
    hf, wf = olm.bf16_to_f64(h), olm.bf16_to_f64(w)
    assert set(np.unique(hf * 8)).issubset(set(range(-8, 9)))
    assert set(np.unique(wf * 256)).issubset(set(range(-8, 9)))
