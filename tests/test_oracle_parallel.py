"""The oracle split over worker processes gives exactly what the single-process oracle gives
(the pool is test infrastructure; the full-size GPU parity tests and the CPU baselines use it)."""
import numpy as np

import oracle
from diffusion_lm_decoding_isd_b300.synthetic import ForwardStream
from oracle.parallel import OraclePool


def test_pool_equals_the_serial_oracle():
    B, N, V = 7, 3, 700
    gen = ForwardStream(B, N, V, 2.0, 0.5, 5, "bf16")
    h0, h1 = gen.next(), gen.next()
    rng = np.random.default_rng(3)
    pend = rng.integers(0, V, size=(B, N - 1)).astype(np.int32)
    pend[1] = -1                                   # a sequence without pending tokens
    pq = rng.uniform(0.01, 1.0, size=(B, N - 1)).astype(np.float32)
    pq[1] = 0.0
    with OraclePool(workers=3) as pool:
        for greedy, T in ((0, 0.8), (1, 1.0), (2, 1.0)):
            prev = None if greedy == 2 else h0
            want = oracle.isd_step(h1, prev, pend, pq, N, T, greedy, 99, 4)
            got = pool.isd_step(h1, prev, pend, pq, N, T, greedy, 99, 4)
            for k in want:
                np.testing.assert_array_equal(np.asarray(got[k]), np.asarray(want[k]), err_msg="%s mode %d" % (k, greedy))
