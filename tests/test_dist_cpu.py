"""bench.py's multi-rank bookkeeping (replicas, one per rank) under gloo on CPU:
barrier, max-over-ranks step time, whole-job weak-scaling throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    assert bench.dist_env() == (ws, rank, rank)
    bench.barrier(ws)
    step_ms = 1.0 + rank  # rank r is slower
    worst = bench.allreduce_max(step_ms, ws, torch.device("cpu"))
    out[rank] = (worst, bench.whole_job_gbs(10**9, ws, worst))
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1]
        worst, gbs = out[0]
        assert worst == 2.0
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.allreduce_max(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_gbs(2 * 10**9, 1, 1.0) == pytest.approx(2000.0)
