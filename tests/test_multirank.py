"""The multi-GPU path of bench.py is token sharding with no data-path
collective: each rank runs the layer on its own batch, and only the timings
are reduced (max over ranks) at the end.  Tested here with two gloo ranks on
the CPU: the reduction, the whole-job throughput and the per-rank inputs."""
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


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from block_scaled_fp8_router_gb300 import synthetic as S
        total, e2e = bench.reduce_max([10.0 + rank, 20.0 - rank], world)
        cfg = S.CONFIGS["tiny"]
        x = S.make_x(cfg, "cpu", bench.rank_seed(0, rank))
        xs = [torch.empty_like(x) for _ in range(world)]
        dist.all_gather(xs, x)
        q.put((rank, total, e2e, bench.job_throughput(cfg.T, 4, world, total), bool(torch.equal(xs[0], xs[1]))))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, e2e, thr, same in res:
        assert total == 11.0 and e2e == 20.0          # the slowest rank's time, on every rank
        assert thr == pytest.approx(256 * 4 * 2 / 11e-3)  # both ranks' tokens over that time
        assert not same                                # the ranks' batches differ


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_throughput(8192, 10, 1, 100.0) == pytest.approx(819200.0)
