"""Multi-GPU runs are independent replicas (no data exchange on the path); the
only cross-rank logic is the bench's timing: barrier, slowest rank's time, and the
whole-job throughput.  Checked here with two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
    ms = bench.max_over_ranks(local_ms, world)
    value = bench.job_throughput(1e12, world, ms)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_max_time_and_sum_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 15.0
        assert abs(value - 2e12 / 15e-3 / 1e12) < 1e-9


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.job_throughput(2e12, 1, 1.0) - 2000.0) < 1e-9
