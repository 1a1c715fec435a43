"""Pins of the oracle's near-tie outputs, on the CPU.

For every inverse-CDF draw the oracle reports the range [cdf_lo, cdf_hi] of
tokens whose CDF interval comes within near_tol * sum(w) of the draw's target
u * sum(w); the parity rule accepts a GPU token anywhere in that range when the
draw is flagged.  The range is pinned by a closed form (equal weights: token j
owns [j/V, (j+1)/V)) and by monotonicity (the draws at u -+ near_tol give the
range's ends); softmax_prob by closed forms.
"""
import math

import numpy as np
import pytest

import oracle


def _recovery_draws(rows, N, T, u_sample, tol):
    """One step of one sequence without pending tokens: draws at rows N-1..2N-2."""
    R = 2 * N - 1
    us = np.full((1, R), u_sample)
    return oracle.isd_step_u(rows[None], None, [[-1] * (N - 1)], [[0.0] * (N - 1)], N, T, 0, np.zeros((1, R)),
                             us, dtype="f32", near_tol=tol)


@pytest.mark.parametrize("V", [1, 7, 10, 64])
@pytest.mark.parametrize("u", [0.0, 0.123, 0.4567, 0.8765, 1.0 - 2.0**-24])  # no edge at u*V
@pytest.mark.parametrize("tol", [1e-6, 0.0413, 0.0737, 0.3141])
def test_window_of_equal_weights(V, u, tol):
    rows = np.zeros((3, V), dtype=np.float32)  # N = 2: rows 0 (anchor, unread), 1 (bonus), 2 (MASK)
    res = _recovery_draws(rows, 2, 1.0, u, tol)
    for r in (1, 2):
        assert res["tokens_out"][0, 0 if r == 1 else r] == math.floor(u * V)
        # token j owns [j/V, (j+1)/V): the window [u - tol, u + tol] meets the tokens from
        # the lowest j with (j+1)/V > u - tol to the highest j with j/V <= u + tol
        lo = max(0, min(V - 1, math.floor((u - tol) * V)))
        hi = max(0, min(V - 1, math.floor((u + tol) * V)))
        assert (res["cdf_lo"][0, r], res["cdf_hi"][0, r]) == (lo, hi), (res["cdf_lo"], res["cdf_hi"], lo, hi)
        x = u * V
        assert res["cdf_margin"][0, r] == pytest.approx(min(x - math.floor(x), math.floor(x) + 1 - x) / V, abs=1e-12)


def test_window_ends_are_the_draws_at_the_window_ends():
    rng = np.random.default_rng(3)
    for trial in range(200):
        V = int(rng.integers(1, 12))
        rows = (rng.standard_normal((3, V)) * 2).astype(np.float32)
        rows[rng.random((3, V)) < 0.2] = -np.inf
        rows[:, int(rng.integers(0, V))] = 0.5  # at least one finite entry per row
        u = float(rng.integers(0, 1 << 24)) * 2.0**-24
        tol = float(rng.choice([1e-3, 0.02, 0.1]))
        res = _recovery_draws(rows, 2, 0.8, u, tol)
        lo_draw = _recovery_draws(rows, 2, 0.8, max(u - tol, 0.0), tol)["tokens_out"][0]
        hi_draw = _recovery_draws(rows, 2, 0.8, u + tol, tol)["tokens_out"][0]
        for r, pos in ((1, 0), (2, 2)):
            assert res["cdf_lo"][0, r] == lo_draw[pos], (trial, r)
            assert res["cdf_hi"][0, r] == hi_draw[pos], (trial, r)
            assert res["cdf_lo"][0, r] <= res["tokens_out"][0, pos] <= res["cdf_hi"][0, r]
            assert np.isfinite(rows[r, res["cdf_lo"][0, r]]) and np.isfinite(rows[r, res["cdf_hi"][0, r]])


def test_no_window_without_a_draw():
    rows = np.zeros((1, 3, 5), dtype=np.float32)
    res = oracle.isd_step(rows, None, [[-1]], [[0.0]], 2, 1.0, 1, 0, 0, dtype="f32")  # greedy: no draws
    assert (res["cdf_lo"] == -1).all() and (res["cdf_hi"] == -1).all() and (res["cdf_margin"] == -1).all()


def test_softmax_prob_closed_forms():
    row = np.array([0.0, math.log(3.0), -np.inf], dtype=np.float64).astype(np.float32)
    assert oracle.softmax_prob(row, 1.0, 1, "f32") == pytest.approx(0.75, rel=1e-7)
    s3 = math.sqrt(3.0)
    assert oracle.softmax_prob(row, 2.0, 1, "f32") == pytest.approx(s3 / (1 + s3), rel=1e-7)
    assert oracle.softmax_prob(row, 1.0, 2, "f32") == 0.0
    bits = np.array([0x3F80, 0x4000], dtype=np.uint16)  # bf16 1.0 and 2.0
    assert oracle.softmax_prob(bits, 1.0, 0, "bf16") == pytest.approx(1 / (1 + math.e), rel=1e-12)
    with pytest.raises(ValueError):
        oracle.softmax_prob(row, 1.0, 3, "f32")
