"""CPU: the multi-replica host logic of bench.py on two gloo ranks.

The layer shards as independent data-parallel replicas with no exchange step,
so bench.py's only cross-rank operations are a barrier and the max over ranks
of each replica's timed region. The whole-job throughput is the tokens of all
ranks divided by that maximum. Two CPU processes stand in for two GPUs here.
"""
import json
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


def _reference_line(*extra):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        *extra], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_line_on_rank_0():
    """Rank 0 prints one JSON line: the oracle's tokens/s, its own cpu_baseline and e2e, the steps it timed."""
    d = _reference_line("--steps", "4", "--warmup", "5", "--reference-budget", "60")
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["steps"] == 4 and d["steps_requested"] == 4
    assert d["warmup"] == 1 and d["warmup_requested"] == 5  # the oracle has nothing to warm up
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny"


def test_reference_arm_stops_at_its_time_budget():
    """Far more steps than the budget allows: the run stops at the budget and says how many steps it timed."""
    d = _reference_line("--steps", "100000", "--warmup", "3", "--reference-budget", "0.5")
    assert 1 <= d["steps"] < 100000 and d["steps_requested"] == 100000
    assert d["ms_per_step"] * d["steps"] >= 500.0 * 0.5  # it ran up to (about) the budget, not past a few steps
