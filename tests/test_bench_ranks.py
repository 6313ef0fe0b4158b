"""The N-GPU path of bench.py is "replicas only": every rank runs its own
step, and the job's figure is all ranks' work over the slowest rank's time.
Its rank logic (barrier, max over ranks, the aggregate) runs here on two CPU
processes over gloo; no GPU is involved."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world, "cpu")
        mine = 10.0 + 5.0 * rank  # this rank's time, ms
        worst = bench.rank_max(mine, world, "cpu")
        value = bench.replicas_throughput(1000, world, worst)
        bench.rank_barrier(world, "cpu")
        q.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_sum_the_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, worst, value in res:
        assert worst == 15.0  # the slower rank's 15 ms, on both ranks
        assert value == pytest.approx(2 * 1000 / 0.015)  # both ranks' units over it


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max(3.5, 1, "cpu") == 3.5
    bench.rank_barrier(1, "cpu")
    assert bench.replicas_throughput(500, 1, 250.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_0_only():
    """Under torchrun the oracle is timed by rank 0 alone; other ranks exit."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.run_reference(None, 1, 2) == 0


def test_reference_arm_line_on_the_host():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys; tiny workload, no GPU needed."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["warmup"] >= 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
