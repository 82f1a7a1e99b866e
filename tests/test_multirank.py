"""The multi-rank path of bench.py on CPU: world_size-2 gloo ranks, no GPU.

The path has no exchange step (one independent replica per GPU), so the only cross-rank logic
is the timing aggregation: the slowest rank's time and the whole-job throughput."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [3.0, 5.0][rank]
    dist.barrier()
    ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
    gbs = bench.whole_job_gbs(world, 1e9, 10, ms * 1e-3)
    q.put((rank, ms, gbs))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, gbs in res:
        assert ms == pytest.approx(5.0)                    # the slower rank's time
        assert gbs == pytest.approx(2 * 1e9 * 10 / 5e-3 / 1e9)


def test_single_rank_aggregation():
    import bench
    assert bench.max_over_ranks(7.5, None, None) == 7.5
    assert bench.whole_job_gbs(1, 23433216, 100, 1e-3) == pytest.approx(2343.3216)
