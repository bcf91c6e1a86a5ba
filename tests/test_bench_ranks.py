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


def test_gpus_flag_without_a_launcher_starts_one_process_per_rank(monkeypatch):
    """`bench.py --gpus 2` with no WORLD_SIZE in the environment relaunches
    itself as two ranks instead of silently running one."""
    seen = {}
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "launch_replicas", lambda n, argv: seen.update(n=n, argv=argv) or 0)
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert e.value.code == 0 and seen["n"] == 2
    cmd = bench.replica_command(2, seen["argv"], 29999)
    assert "--nproc-per-node=2" in cmd and "--master-addr=127.0.0.1" in cmd
    assert cmd[-4:] == ["--steps", "3", "--warmup", "3"]


def test_replicas_run_as_two_ranks_and_rank0_prints_one_line():
    """The relaunch command itself, on CPU: two ranks of the reference arm; rank
    0 alone prints the JSON line, which reports both ranks."""
    import json
    import subprocess
    cmd = bench.replica_command(2, ["--impl", "reference", "--gpus", "2", "--workload",
                                    "tiny_fp32", "--steps", "3", "--warmup", "3"], _free_port())
    env = dict(os.environ, OMP_NUM_THREADS="1")
    env.pop("WORLD_SIZE", None)
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["impl"] == "reference"
