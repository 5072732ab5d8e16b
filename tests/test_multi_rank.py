"""The N > 1 host path of bench.py on CPU (gloo, world size 2): each rank runs
its own problem, the job's time is the slowest rank's, and the job's bytes are
all ranks' (weak scaling).  No GPU involved."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._pg = dist.group.WORLD
    try:
        local_ms = [40.0, 50.0][rank]          # rank 1 is the slow one
        gbs, job_ms = bench.whole_job_gbs(1e9, 10, world, local_ms)
        bench.barrier()
        results[rank] = (gbs, job_ms, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_ranks_aggregate_on_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    for r in range(2):
        gbs, job_ms, env = res[r]
        assert job_ms == 50.0
        assert gbs == pytest.approx(1e9 * 10 * 2 / 0.05 / 1e9)
        assert env == (2, r, r)


def test_reference_arm_other_ranks_print_nothing(capsys):
    import bench

    class A:
        kv, steps, warmup = 256, 1, 0
    bench.reference_arm(A, 2, 1)
    assert capsys.readouterr().out == ""
