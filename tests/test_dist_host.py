"""The multi-process bookkeeping of bench.py (replicas: barrier, max over
ranks, whole-job aggregate) on two gloo ranks on the host, no GPU."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    try:
        import torch.distributed as dist
        import bench
        ws, r, _ = bench.dist_setup()
        bench.barrier(ws)
        ms = bench.max_over_ranks(10.0 * (rank + 1), ws)       # rank 1 is the slower one
        rate = bench.whole_job_rate(65536, ms, ws)
        q.put((rank, ws, r, dist.get_backend(), ms, rate))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, *rest in got:
        assert rest[0] != "error", rest
        ws, r, backend, ms, rate = rest
        assert (ws, r, backend) == (2, rank, "gloo")
        assert ms == pytest.approx(20.0)
        assert rate == pytest.approx(2 * 65536 / 0.020)
