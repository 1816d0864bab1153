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


def test_shard_ranges_tile_the_vocabulary():
    """detlm_shard_range (host code of the library, no GPU): the P ranges are
    contiguous, cover [0, V), start on 256-entry tiles, and are the tiles of
    the leaves [128 r / P, 128 (r + 1) / P) of the log-sum-exp tree."""
    from invariant_output_head_gb300 import DetlmError, binding as bd
    for V in (1, 255, 256, 257, 1000, 32000, 151936, 152064, 128256, 2 ** 31 - 1):
        n = (V + 255) // 256
        leaf_lo = [g * n // 128 for g in range(129)]
        for P in (1, 2, 4, 8, 16, 128):
            prev = 0
            for r in range(P):
                a, b = bd.detlm_shard_range(V, P, r)
                assert a == prev and a % 256 == 0 and b >= a
                assert a == 256 * leaf_lo[r * (128 // P)]
                assert b == min(V, 256 * leaf_lo[(r + 1) * (128 // P)])
                prev = b
            assert prev == V
    for V, P, r in ((1000, 3, 0), (1000, 0, 0), (1000, 256, 0), (1000, 4, 4), (0, 1, 0),
                    (1000, 4, -1)):
        with pytest.raises(DetlmError):
            bd.detlm_shard_range(V, P, r)


def _shard_record(case, V, P, r):
    """Shard r's records [B, 4] (int32 words) built from the oracle's logits of
    its rows: greedy (max as f32, lowest global index, runner-up as f32) and
    the log-prob target flag and target logit."""
    import numpy as np
    import oracle
    from invariant_output_head_gb300 import binding as bd
    v0, v1 = bd.detlm_shard_range(V, P, r)
    z, _ = oracle.logits_float(oracle.decode(case["W"][v0:v1], "bf16"),
                               oracle.decode(case["h"], "bf16"))
    tok, m, s = oracle.top2(z)
    t = case["targets"]
    here = (t >= v0) & (t < v1)
    zt = np.where(here, z[np.arange(z.shape[0]), np.clip(t - v0, 0, v1 - v0 - 1)], 0.0)
    rec = np.zeros((z.shape[0], 4), dtype=np.int32)
    rec[:, 0] = m.astype(np.float32).view(np.int32)
    rec[:, 1] = (tok + v0).astype(np.int32)
    rec[:, 2] = s.astype(np.float32).view(np.int32)
    rec[:, 3] = np.where(here, zt, 0.0).astype(np.float32).view(np.int32)
    return rec, here


def _shard_rank_main(rank, world, port, q):
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import synth
    from invariant_output_head_gb300 import binding as bd
    V, d, B = 3000, 64, 6
    case = synth.small_float(31, V, d, B, n_ties=2)
    rec, _ = _shard_record(case, V, world, rank)
    got = bd.gather_records(torch.from_numpy(rec)).numpy()       # [P, B, 4]
    ok = got.shape == (world, B, 4)
    # shard-major, in rank order: record k is the one rank k built
    for k in range(world):
        ok = ok and (got[k] == _shard_record(case, V, world, k)[0]).all()
    # merging the gathered records (exact rule: value desc, index asc) gives
    # the oracle's token over the whole vocabulary; exactly one shard holds
    # each row's target
    z, _ = oracle.logits_float(oracle.decode(case["W"], "bf16"), oracle.decode(case["h"], "bf16"))
    m = got[:, :, 0].view(np.float32)
    idx = got[:, :, 1]
    best = np.lexsort((idx, -m), axis=0)[0]                    # per row: winning shard
    tok = idx[best, np.arange(B)]
    ok = ok and (tok == oracle.top2(z.astype(np.float32).astype(np.float64))[0]).all()
    holders = np.stack([_shard_record(case, V, world, k)[1] for k in range(world)])
    ok = ok and (holders.sum(axis=0) == 1).all()
    q.put((rank, bool(ok)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_gather_shard_records_in_rank_order():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, True), (1, True)]
