"""The multi-rank plumbing of bench.py (replicas, barrier, max-over-ranks timing, whole-job
aggregate) on CPU with two gloo ranks; and the reference arm's rank rule."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = bench.dist_env()
    bench.dist_init(w)
    bench.dist_barrier(w)
    ms = 10.0 * (rank + 1)                       # rank 1 is the slower replica
    ms_max = bench.dist_max(ms, w)
    out[rank] = (r, w, ms_max, bench.whole_job_value(w, 4096, 5, ms_max))
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_aggregate():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][:3] == (0, 2, 20.0) and res[1][:3] == (1, 2, 20.0)
    # both ranks processed 4096 tokens per step for 5 steps in at most 20 ms
    assert res[0][3] == pytest.approx(2 * 4096 * 5 / 0.020)


def test_single_rank_defaults():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.dist_max(3.5, 1) == 3.5
    assert bench.whole_job_value(1, 4096, 10, 40.0) == pytest.approx(4096 * 10 / 0.040)
