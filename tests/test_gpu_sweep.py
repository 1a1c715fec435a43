"""Acceptance / stride sweep on the GPU path (a reduced copy of bench.py --sweep): measured
tokens per forward against the closed form TPF = (2+p+...+p^(N-2)) / (2-p^(N-1)) at the
measured per-token acceptance p_hat ("Speedup Factor Explorer", de.news.hada.io).

The closed form is exact for independent acceptances with a constant probability; the
synthetic forwards give every pending token its own probability, so only a loose agreement is
asserted, together with what must hold exactly: 1 <= TPF <= N and p_hat falling as the anchor
noise grows."""
import pytest

import bench

pytestmark = pytest.mark.gpu


def test_sweep_tracks_closed_form():
    rows = bench.run_sweep(None, 0, 0, steps=96, Ns=(2, 4, 8), sigmas=(0.1, 1.0))
    by = {(r["N"], r["sigma_n"]): r for r in rows}
    for r in rows:
        assert 1.0 <= r["tpf"] <= r["N"], r
        assert abs(r["rel_diff"]) < 0.08, r
    for N in (2, 4, 8):
        assert by[(N, 0.1)]["p_hat"] > by[(N, 1.0)]["p_hat"]
        assert by[(N, 0.1)]["tpf"] > by[(N, 1.0)]["tpf"]
