"""Host-side multi-process logic of bench.py on CPU: two gloo ranks, each with its own
batch seed; the job's time and every stage's time are the slowest rank's (max over ranks),
the whole-job rate counts every rank's tokens, only rank 0 prints, and `--gpus 2` starts
the two ranks itself.  No GPU is used."""
import json
import os
import socket
import subprocess
import sys

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
    stages = bench.max_stage_times({"gemm": 2.0 - rank, "combine": 0.1 * (rank + 1)}, w)
    printed = bench.emit({"rank": rank}, rank)
    out[rank] = (bench.max_over_ranks(mine, w), bench.rank_seed(0, rank), stages, printed)
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
    assert res[0][2] == res[1][2] == {"gemm": 2.0, "combine": 0.2}
    assert res[0][3] is True and res[1][3] is False


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(8192, 4, 8.0) == 8192 * 4 / 8e-3


def test_gpus_flag_starts_the_ranks_itself():
    """`bench.py --gpus 2` outside torchrun runs two ranks of one node (127.0.0.1
    rendezvous, gloo for the CPU reference arm): exactly one JSON line, from rank 0, with
    n_gpus 2."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR",
                                                            "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1", "--ref-tokens", "2"],
                       capture_output=True, text=True, timeout=600, cwd=root, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def test_single_process_defaults():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.25, 1) == 3.25
