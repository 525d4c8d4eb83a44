"""The multi-GPU path is replicas only (every rank runs its own copy of the
step; no data-path collective). Its host logic - gathering every rank's
timings and reducing them to whole-job numbers - runs here as world-size-2
gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r processed 1e9 * (r + 1) draft bytes in (r + 1) ms, verify 3e9 bytes in 2 ms
    stats = bench.gather_stats((1e9 * (rank + 1), 1.0 + rank, 3e9, 2.0, 10.0 + rank), world)
    agg = bench.replica_aggregate(stats)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, stats, agg))


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, stats, agg in res:
        assert len(stats) == 2
        # whole-job bytes (1e9 + 2e9) over the slowest rank's 2 ms
        assert agg["gemv_gbs"] == pytest.approx(3e9 / 2e-3 / 1e9)
        assert agg["gemm_gbs"] == pytest.approx(6e9 / 2e-3 / 1e9)
        assert agg["ms_per_step"] == pytest.approx(11.0)


def test_replica_aggregate_single_rank_is_identity():
    import bench
    agg = bench.replica_aggregate([(2e9, 4.0, 6e9, 3.0, 7.5)])
    assert agg["gemv_gbs"] == pytest.approx(500.0)
    assert agg["gemm_gbs"] == pytest.approx(2000.0)
    assert agg["ms_per_step"] == 7.5
    assert torch.__version__
