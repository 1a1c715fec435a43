"""The oracle's pins are sharp: plant one plausible mistake at a time in a copy
of the oracle source (on the CPU), rebuild it, and check that some pin fails.

Nothing here touches the committed oracle; each mutant is a temporary build.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import build as oracle_build
from test_oracle_enumeration import _first_token_law, _rows
from test_oracle_greedy import ToyAR, run_isd
from test_oracle_tpf import closed_form_tpf, simulate_tpf

# (name, text in isd_oracle.c, replacement)
MUTANTS = [
    ("anchor_row_off_by_one",
     "pout[i - 1] = P[(size_t)(i - 1) * V + pend[i - 1]];",
     "pout[i - 1] = P[(size_t)(i) * V + pend[i - 1]];"),
    ("residual_sign_flipped", "double d = Pk[j] - Q[j];", "double d = Q[j] - Pk[j];"),
    ("residual_q_from_wrong_row", "qoff = seq_off + (size_t)(N + K) * V;",
     "qoff = seq_off + (size_t)(N - 1 + K) * V;"),
    ("no_replacement_token", "tok[n_emit++] = y;\n                propose = 0;",
     "propose = 0;"),
    ("proposals_kept_after_rejection", "propose = 0; /* the proposals", "propose = 1; /* the proposals"),
    ("acceptance_ratio_inverted", "const double ratio = pout[i - 1] / (double)pq[i - 1];",
     "const double ratio = (double)pq[i - 1] / pout[i - 1];"),
    ("philox_constant_typo", "0xD2511F53u", "0xD2511F55u"),
    ("philox_key_not_bumped", "k0 += PHILOX_W0;", "k0 += 0;"),
    ("uniform_23_bits", "return ldexp((double)(w >> 8), -24);", "return ldexp((double)(w >> 9), -23);"),
    ("argmax_highest_index_on_ties", "if (x > bv) { bv = x; best = j; }",
     "if (x >= bv) { bv = x; best = j; }"),
    ("inverse_cdf_non_strict", "if (pick < 0 && C > target) {", "if (pick < 0 && C >= target) {"),
    ("temperature_ignored", "double z = logit_at(base, dtype, off + (size_t)j) / T;\n        P[j]",
     "double z = logit_at(base, dtype, off + (size_t)j);\n        P[j]"),
    ("bonus_from_mask_row", "y = inverse_cdf(P + (size_t)(N - 1) * V, V, us[N - 1], near_tol,",
     "y = inverse_cdf(P + (size_t)(N) * V, V, us[N - 1], near_tol,"),
    ("proposal_q_not_saved", "nq[j - 1] = P[(size_t)r * V + x];", "nq[j - 1] = 1.0;"),
    # argmax proposals with sampled verification (greedy = 2)
    ("argmax_residual_keeps_x", "Q[pend[K]] = 1.0;", "Q[pend[K]] = 0.0;"),
    ("argmax_proposal_q_not_one", "nq[j - 1] = 1.0; /* an argmax proposal is a point mass */",
     "nq[j - 1] = 0.5; /* an argmax proposal is a point mass */"),
    ("argmax_proposals_sampled", "if (greedy >= 1) {", "if (greedy == 1) {"),
]


def _kat_ok():
    here = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    for line in open(here):
        if line.strip() and not line.startswith("#"):
            w = [int(x, 16) for x in line.split()]
            if oracle.philox4x32_10(w[0:4], w[4:6]) != w[6:10]:
                return False
    return oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24 and oracle.uniform(0x100) == 2.0 ** -24


def _enum_ok():
    rng = np.random.default_rng(31)
    for N, V, T in ((2, 5, 0.7), (3, 4, 1.0)):
        prev = _rows(rng, N, V)
        cur = _rows(rng, N, V)
        half = V // 2
        for disjoint in (False, True):
            pv, cu = prev.copy(), cur.copy()
            if disjoint:
                cu[0, :half] = -np.inf
                pv[N, half:] = -np.inf
            try:
                law = _first_token_law(pv, cu, N, T)
            except AssertionError:
                return False
            x = cu[0].astype(np.float64) / T
            p = np.exp(x - x.max())
            p /= p.sum()
            got = np.array([law.get(y, 0.0) for y in range(V)])
            if np.max(np.abs(got - p)) > 2e-6:
                return False
            if disjoint and any(law.get(y, 0.0) != 0.0 for y in range(half)):
                return False
    return True


def _tpf_ok():
    for N, alpha in ((4, 0.9), (2, 0.5)):
        tpf, se = simulate_tpf(N, alpha, B=600, steps=60, burn=10)
        if abs(tpf - closed_form_tpf(N, alpha)) > 4 * se:
            return False
    return True


def _greedy_ok():
    rows = np.zeros((1, 3, 6), dtype=np.float32)
    rows[0, 1, [2, 4]] = 5.0
    rows[0, 2, [1, 3]] = 7.0
    res = oracle.isd_step(rows, None, [[-1]], [[0.0]], 2, 1.0, True, 0, 0, dtype="f32")
    if res["tokens_out"][0].tolist() != [2, -1, 1]:
        return False
    f = ToyAR(8, 30)
    stream, _ = run_isd(f, 3, 30, 30, 0.8, seed=1)
    return stream == f.greedy([], 30)


def _sampled_low_t_ok():
    f = ToyAR(77, 30, scale=3.0)
    a, _ = run_isd(f, 4, 30, 30, 1.0, seed=3, greedy=True)
    b, _ = run_isd(f, 4, 30, 30, 1.0, seed=3, greedy=False, T=1e-4)
    return a == b


def _argmax_mode_ok():
    rng = np.random.default_rng(41)
    for N, V, T in ((2, 5, 1.0), (3, 4, 0.8)):
        prev = _rows(rng, N, V)
        cur = _rows(rng, N, V)
        law = _first_token_law(prev, cur, N, T, mode=2)
        x = cur[0].astype(np.float64) / T
        p = np.exp(x - x.max())
        p /= p.sum()
        got = np.array([law.get(y, 0.0) for y in range(V)])
        if np.max(np.abs(got - p)) > 2e-6:
            return False
    return True


PINS = [_kat_ok, _enum_ok, _tpf_ok, _greedy_ok, _sampled_low_t_ok, _argmax_mode_ok]


def _build_mutant(tmpdir, old, new):
    src = open(oracle_build.SRC).read()
    assert src.count(old) == 1, "mutation anchor must occur exactly once: %r" % old
    path = os.path.join(tmpdir, "isd_oracle_mutant.c")
    with open(path, "w") as fh:
        fh.write(src.replace(old, new))
    lib = os.path.join(tmpdir, "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", lib, path, "-lm"],
                   check=True)
    return lib


def test_pins_pass_on_the_real_oracle():
    assert all(pin() for pin in PINS)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    lib = _build_mutant(str(tmp_path), old, new)
    with oracle.using_library(lib):
        results = {}
        for pin in PINS:
            try:
                results[pin.__name__] = bool(pin())
            except (AssertionError, ValueError, IndexError):
                results[pin.__name__] = False
    assert not all(results.values()), "no pin caught mutant %s: %s" % (name, results)
