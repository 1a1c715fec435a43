"""Host logic of the multi-GPU replicas, on CPU: two gloo ranks (127.0.0.1).

Sequences are independent, so bench.py runs one replica of the workload per rank with no
data-path collective; the process group only carries the barrier and the host reductions of
the timings (max over ranks) and of the emitted tokens (sum over ranks).  A rank that is not
rank 0 prints nothing, and the reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.barrier(world)
    # per-rank timings and token counts of a replica run
    elapsed = [12.5, 20.0][rank]
    tokens = [1000, 3000][rank]
    out[rank] = (bench.max_over_ranks(elapsed, world), bench.sum_over_ranks(tokens, world),
                 bench.run_reference(bench.parse_args([]), {}, rank, world) is None if rank else True)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_timings_and_tokens():
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    for rank in (0, 1):
        t_max, tok_sum, ref_none = out[rank]
        assert t_max == 20.0          # the job's time is the slowest replica's
        assert tok_sum == 4000        # value = tokens of all replicas / that time
        assert ref_none               # the reference arm runs on rank 0 only
