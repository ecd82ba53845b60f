"""The bench's multi-rank path on CPU: two gloo ranks, each timing its own
replica, agree on the whole-job throughput computed from the slowest rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [10.0, 12.5][rank]  # rank 1 is the slower replica
    m = bench.max_over_ranks(local_ms, world, "cpu")
    results[rank] = (m, bench.whole_job_tflops(1e12, 4, world, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_use_the_slowest_replica():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0] == results[1]
    m, tflops = results[0]
    assert m == pytest.approx(12.5)
    # 2 ranks x 4 steps x 1 TFLOP in 12.5 ms
    assert tflops == pytest.approx(2 * 4 * 1.0 / 12.5e-3)


def test_single_rank_is_unchanged():
    import bench

    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.whole_job_tflops(2e12, 5, 1, 10.0) == pytest.approx(1000.0)
