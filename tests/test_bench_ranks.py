"""The multi-GPU bench path on CPU: N replicas (one per rank, no data-path
collective) are timed with a barrier and the slowest rank's time; the
whole-job value counts every rank's bytes.  Two gloo ranks stand in for two
GPUs here."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], torch.device("cpu"), world)
        value = bench.whole_job_gbs(1_000_000_000, world, slowest)
        # the reference arm: rank 0 alone runs it, the other ranks return nothing
        ref = None if rank == 0 else bench.run_reference(None, world, rank)
        out_q.put((rank, slowest, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.010, 0.025]
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, ref in results:
        assert slowest == pytest.approx(0.025)
        assert value == pytest.approx(2 * 1.0 / 0.025)      # 2 ranks x 1 GB / slowest time
        if rank != 0:
            assert ref is None


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, torch.device("cpu"), 1) == 3.5
    assert bench.whole_job_gbs(2_000_000_000, 1, 0.5) == pytest.approx(4.0)
