"""The multi-rank path of bench.py on CPU (gloo, world size 2): every rank
draws its own seeded problem, the job time is the slowest rank's, and the
reported throughput counts the units of all ranks.  The KDA work itself is
per (sequence, head) and exchanges nothing between ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        my_ms = 1.0 + 2.0 * rank  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(my_ms, ws, torch.device("cpu"))
        seed = bench.rank_seed(7, rank)
        dist.barrier()
        q.put((rank, job_ms, seed, bench.dist_info()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.0, 3.0]          # max over ranks, seen by every rank
    assert res[0][2] != res[1][2]                      # independent problems per rank
    assert [r[3] for r in res] == [(2, 0, 0), (2, 1, 1)]
    # whole-job throughput: units of all ranks over the slowest rank's time
    assert bench.aggregate_throughput(1000, ws, 3.0) == pytest.approx(2000 / 3e-3)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    assert bench.rank_seed(3, 0) == 3
