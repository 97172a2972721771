"""The multi-GPU path is replicas only: each rank runs the whole hot path on
its own GPU and the benchmark reports all ranks' tokens over the slowest
rank's time. The cross-rank logic (barrier, max over ranks, whole-job
throughput) is tested here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    rank_ms = [120.0, 150.0][rank]              # rank 1 is the slowest replica
    slow = bench.max_over_ranks(rank_ms, world)
    value = bench.replica_throughput(8192, 10, rank_ms, world)
    q.put((rank, slow, value))
    dist.destroy_process_group()


def test_replicas_report_slowest_rank_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slow, value in res:
        assert slow == 150.0
        assert value == pytest.approx(2 * 8192 * 10 / 0.150)
