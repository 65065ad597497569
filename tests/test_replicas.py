"""The multi-process path of bench.py on CPU: one replica per rank (the GEMM
and attention calls shard into independent problems, so there is no
data-path collective), the timed region closed by the slowest rank, and the
whole-job throughput counting every rank's work.  Two gloo ranks on
127.0.0.1."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        # each rank's own elapsed time; the job's is the largest
        mine = 10.0 + 5.0 * rank
        dist.barrier()
        job_ms = bench.max_over_ranks(mine, ws, torch.device("cpu"))
        value = bench.job_throughput(2.0e12, ws, 4, job_ms)
        out.put((r, local, ws, job_ms, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_over_ranks_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and [r[1] for r in res] == [0, 1]
    for (_, _, ws, job_ms, value) in res:
        assert ws == 2
        assert job_ms == 15.0                          # the slowest rank's time
        # both ranks' 4 steps of 2e12 units in 15 ms: 1066.67 tera-units/s
        assert value == pytest.approx(2 * 2.0e12 * 4 / 15e-3 / 1e12)


def test_one_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(7.5, 1, torch.device("cpu")) == 7.5
    assert bench.job_throughput(1.0e12, 1, 10, 1000.0) == pytest.approx(10.0)
