"""bench.py's multi-rank helpers with gloo, world size 2, on CPU: each rank
builds its own replica (independent seed, same shape recipe), and the step
time reported is the maximum over ranks."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    case = bench.replica_case("c0", rank)
    mx = bench.all_max(float(rank + 1) * 1.5, world)
    bench.barrier(world)
    out[rank] = (float(case.q.double().sum()), mx, case.q.shape, tuple(case.context_lens.tolist()))
    dist.destroy_process_group()


def test_two_rank_replicas_and_max():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        r0, r1 = out[0], out[1]
    assert r0[1] == r1[1] == 3.0            # max over ranks
    assert r0[2] == r1[2]                    # same shapes
    assert r0[3] == r1[3] == (7, 16, 33, 50)  # the tiny workload's lengths are fixed
    assert r0[0] != r1[0]                    # independent values per replica
