"""CPU: the multi-replica host logic of bench.py on two gloo ranks.

The layer shards as independent data-parallel replicas with no exchange step,
so bench.py's only cross-rank operations are a barrier and the max over ranks
of each replica's timed region. The whole-job throughput is the tokens of all
ranks divided by that maximum. Two CPU processes stand in for two GPUs here.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 200.0][rank]           # the second replica is the slower one
    dist.barrier()
    ms = bench.max_over_ranks(local_ms, world, "cpu")
    v = bench.job_tokens_per_s(64, world, 10, ms)
    dist.destroy_process_group()
    q.put((rank, ms, v))


def test_max_over_ranks_and_job_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, v in res:
        assert ms == 200.0                       # every rank sees the slowest replica's time
        assert v == pytest.approx(64 * 2 * 10 / 0.2)   # all ranks' tokens over that time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(64, 1, 1000, 500.0) == pytest.approx(128000.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""
