"""Multi-rank logic of bench.py on CPU with gloo, world size 2: every rank
draws an independent batch of the same shape, the job time is the slowest
rank's, and the job value counts all ranks' tokens."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, REPO)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = bench.rank_batch("tinyllama", rank)
    fake_ms = 10.0 + 5.0 * rank
    job_ms = bench.max_over_ranks(fake_ms, dist)
    gathered = [None] * world
    dist.all_gather_object(gathered, (b.seed, b.seq_lens.tolist(), b.block_table.shape))
    out[rank] = (job_ms, bench.job_tokens_per_s(world, b.num_tokens, job_ms), gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        job_ms, value, gathered = res[rank]
        assert job_ms == 15.0                         # the slower rank's time
        assert abs(value - 2 * 64 / 15e-3) < 1e-6     # both ranks' 64 tokens each
        (s0, l0, sh0), (s1, l1, sh1) = gathered
        assert s0 != s1 and l0 != l1                  # independent problems
        assert sh0[0] == sh1[0] == 64                 # same shape per rank


def test_single_rank_reduction_is_identity():
    import sys
    sys.path.insert(0, REPO)
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert np.isclose(bench.job_tokens_per_s(1, 256, 0.5), 512000.0)
