"""N > 1 host logic on CPU: row sharding and the max-over-ranks step time,
run as two gloo ranks (no GPU, no data-path collective)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from mx_scale_reusing_gb300 import shard


@pytest.mark.parametrize("T,world", [(0, 2), (1, 2), (7, 2), (65536, 2), (65537, 3), (5, 8)])
def test_row_ranges_partition_the_batch(T, world):
    ranges = [shard.row_range(T, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0 and a0 <= a1
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_bad_arguments():
    with pytest.raises(ValueError):
        shard.row_range(8, 2, 2)
    with pytest.raises(ValueError):
        shard.row_range(8, 0, 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T = 1001
        r0, r1 = shard.row_range(T, rank, world)
        # each rank "processes" its rows; the slow rank decides the step time
        step_ms = 1.0 + rank * 2.5
        out[rank] = (r0, r1, shard.max_over_ranks(step_ms), shard.rank_seed(3, rank))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][:2] == (0, 501) and res[1][:2] == (501, 1001)
    assert res[0][2] == res[1][2] == 3.5
    assert res[0][3] != res[1][3]
