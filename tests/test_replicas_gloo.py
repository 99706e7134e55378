"""The N > 1 path of bench.py (independent replicas, one rank per GPU) on CPU with two gloo
ranks: the timing rule (maximum over ranks), distinct per-rank workloads, the whole-job rate,
and the reference arm running on rank 0 only."""
import contextlib
import io
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        seed = bench.replica_seed(1003, rank)
        out = io.StringIO()
        if rank != 0:
            # the reference arm under torchrun: rank 0 alone runs and prints
            args = type("A", (), {"steps": 1, "warmup": 0, "gpus": world})()
            with contextlib.redirect_stdout(out):
                bench.run_reference(args)
        dist.barrier()
        q.put((rank, t, seed, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    times = [r[1] for r in res]
    assert times == [15.0, 15.0]                       # every rank sees the slowest rank
    assert len({r[2] for r in res}) == world           # a distinct workload per replica
    assert res[1][3] == ""                             # rank 1 prints nothing
    import bench
    # 2 ranks x 3840 rows x 10 steps in 15 ms
    assert bench.whole_job_rate(3840, 10, world, 15.0) == pytest.approx(2 * 3840 * 10 / 0.015)
