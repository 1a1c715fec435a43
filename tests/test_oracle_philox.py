"""Pins of the oracle's counter-based generator and uniform construction."""
import os

import numpy as np

import oracle


def _read_kat(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "philox4x32_10_kat.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = [int(x, 16) for x in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answer_vectors(golden_dir):
    kat = _read_kat(golden_dir)
    assert len(kat) == 3
    for ctr, key, expect in kat:
        assert oracle.philox4x32_10(ctr, key) == expect


def test_uniform_construction_edges():
    # top 24 bits of the word times 2^-24: [0, 1 - 2^-24], exact in fp32
    assert oracle.uniform(0) == 0.0
    assert oracle.uniform(0xFF) == 0.0
    assert oracle.uniform(0x100) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform(0x80000000) == 0.5
    for w in (0x12345678, 0xDEADBEEF, 0x00ABCDEF):
        u = oracle.uniform(w)
        assert float(np.float32(u)) == u


def test_row_uniforms_use_counter_layout():
    # counter = (step lo, step hi, seq, row), key = (seed lo, seed hi);
    # word 0 -> acceptance uniform, word 1 -> sampling uniform
    seed = 0x0123456789ABCDEF
    step = 0x00000002_00000007
    w = oracle.philox4x32_10([step & 0xFFFFFFFF, step >> 32, 5, 3],
                             [seed & 0xFFFFFFFF, seed >> 32])
    ua, us = oracle.row_uniforms(seed, step, 5, 3)
    assert ua == (w[0] >> 8) * 2.0 ** -24
    assert us == (w[1] >> 8) * 2.0 ** -24


def test_uniforms_are_uniform_and_decorrelated():
    # a statistical sanity check of the stream the step draws from
    vals = np.array([oracle.row_uniforms(7, t, b, r)
                     for t in range(40) for b in range(10) for r in range(7)])
    n = len(vals)
    for col in range(2):
        u = np.sort(vals[:, col])
        ks = np.max(np.abs(u - (np.arange(1, n + 1) - 0.5) / n))
        assert ks < 1.63 / np.sqrt(n) + 0.5 / n  # KS test at about 1%
    assert abs(np.corrcoef(vals[:, 0], vals[:, 1])[0, 1]) < 0.1
