"""Multi-rank logic of the benchmark on CPU (gloo, world size 2).

The path shards by tokens into independent problems: each rank draws its own
replica of the workload, the job time is the slowest rank's, and the job
rate counts every rank's units.  No data-path collective is involved; the only
collective is the max over ranks of the timing."""
import os
import socket

import pytest
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
    try:
        import bench
        t = bench.max_over_ranks(1.5 + rank, world, "cpu")
        seed = bench.workload_seed("bf16_prefill", rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        q.put((rank, t, seeds))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_distinct_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    results = sorted(q.get() for _ in range(world))
    for rank, t, seeds in results:
        assert t == pytest.approx(2.5)           # max over ranks
        assert len(set(seeds)) == world          # each rank its own replica


def test_job_throughput_is_weak_scaling():
    import bench
    # 2 ranks, 10 units each per step, 3 steps, slowest rank 2 s -> 30 units/s
    assert bench.job_throughput(10, 2, 3, 2.0) == pytest.approx(30.0)
    assert bench.job_throughput(10, 1, 3, 1.0) == pytest.approx(30.0)


def _bench(*argv):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *argv],
                          capture_output=True, text=True, timeout=600, env=env, cwd=root)


def test_bench_spawns_its_ranks_when_run_without_a_launcher():
    """bench.py --gpus 2 with no WORLD_SIZE starts two ranks itself (gloo for
    the oracle arm here); rank 0 prints one line that counts both."""
    import json
    r = _bench("--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "1",
               "--warmup", "1", "--ref-tokens", "2")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["impl"] == "reference"


def test_bench_refuses_more_gpus_than_visible():
    import torch
    n = torch.cuda.device_count()
    r = _bench("--gpus", str(n + 1), "--steps", "1", "--warmup", "3")
    assert r.returncode != 0
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
