"""The multi-rank logic of bench.py on CPU: two gloo ranks, each timing its
own replica of the workload.  Every rank must end up with the max time over
ranks, and the whole-job throughput counts the bytes of all ranks."""
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


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        w, r, local = bench.dist_setup()
        assert (w, r, local) == (world, rank, rank)
        m = bench.max_over_ranks(times[rank], "cpu")
        out[rank] = (m, bench.job_gbs(w, 327_680_000, 100, m))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    times = [4.0, 5.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 5.5
    # 2 replicas x 100 steps x 327.68 MB in 5.5 ms
    assert out[0][1] == pytest.approx(2 * 327_680_000 * 100 / 5.5e-3 / 1e9)


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_gbs(1, 8, 1, 1.0) == pytest.approx(8e-6)
