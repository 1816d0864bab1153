"""The benchmark's multi-rank host logic on two gloo ranks (CPU only): the
barrier, the max-over-ranks timing, and the whole-job throughput of weak
scaling (every rank runs the same per-GPU workload, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    elapsed = [12.5, 20.0][rank]
    m = bench.max_over_ranks(elapsed, world)
    v = bench.job_rows_per_s(16, 100, world, m)
    q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, m, v in res:
        assert m == 20.0                               # the slowest rank
        assert v == pytest.approx(16 * 100 * 2 / 0.020)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_rows_per_s(16, 10, 1, 1000.0) == 160.0
