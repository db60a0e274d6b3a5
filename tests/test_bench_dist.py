"""Host-side multi-process logic of bench.py on CPU: two gloo ranks, each with its own
batch seed; the job's time is the slowest rank's (max over ranks) and the weights' seed is
shared.  No GPU is used."""
import os
import socket

import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    mine = 1.5 + rank                      # rank 1 is the slow one
    out[rank] = (bench.max_over_ranks(mine, w), bench.rank_seed(0, rank))
    bench.barrier(w)
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_draw_their_own_batches():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5
    assert res[0][1] != res[1][1]


def test_single_process_defaults():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25
