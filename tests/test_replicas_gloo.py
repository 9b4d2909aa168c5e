"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks.

The layer shards by tokens with no exchange step, so N GPUs run N independent replicas; the
only cross-rank operations are the timing barrier and the max over ranks.  This test runs two
gloo ranks that each "time" a different amount of work and checks that both see the slowest
rank's time and that the job throughput counts every rank's units over that time.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 * (rank + 1)                  # rank 1 is the slow replica
    dist.barrier()
    ms = bench.max_over_ranks(local_ms, world)
    tput = bench.job_throughput(4096 * 5, world, ms / 1e3)
    out[rank] = (ms, tput)
    dist.barrier()
    dist.destroy_process_group()
    del torch


@pytest.mark.timeout(120)
def test_two_gloo_replicas_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0][0] == out[1][0] == 20.0
    assert out[0][1] == out[1][1] == pytest.approx(4096 * 5 * 2 / 0.020)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(100, 1, 0.5) == 200.0


@pytest.mark.timeout(600)
def test_bench_gpus_2_launches_two_ranks_and_prints_one_line():
    """`bench.py --gpus 2` without a launcher environment starts two ranks itself (as
    torch.distributed.run would, rendezvous on 127.0.0.1); on the reference arm rank 0 alone
    runs and prints, the other rank exits 0 without work."""
    import json
    import subprocess
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=540, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
