"""The bench's multi-GPU path on the CPU: two gloo ranks.  Each rank owns its
own heads (inputs seeded by rank, no collective on the data path); the step time
reported is the max over ranks and the work is the sum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from optimal_tiling_gb300 import inputs
    ws, r, local = bench._dist()
    d = bench._init_pg(ws, "gloo")
    assert d is not None and ws == world and r == rank
    mx = bench._max_over_ranks(d, 10.0 + rank)
    sm = bench._sum_over_ranks(d, 1.0 + rank)
    x = inputs.make_inputs(1, 1, 128, 8, torch.float32, seed=rank, with_do=False)
    gathered = [torch.zeros(128 * 8) for _ in range(world)]
    dist.all_gather(gathered, x["q"].flatten())
    distinct = not torch.equal(gathered[0], gathered[1])
    out[rank] = (mx, sm, distinct)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()   # no fork of a process that already runs threads
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        mx, sm, distinct = out[rank]
        assert mx == 11.0          # max over ranks of 10 + rank
        assert sm == 3.0           # sum over ranks of 1 + rank
        assert distinct            # each rank's heads are its own data
