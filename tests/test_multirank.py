"""The benchmark's multi-rank host logic on CPU: two gloo ranks, barrier and max-over-ranks.

Every GPU rank runs an independent replica of the workload (no collective on the data path); the
only collectives are the timing barrier and the max reduction of the per-rank step time, and the
whole-job value is the sum of the ranks' tokens over that max time."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist(torch)
    d.init("gloo")
    d.barrier()
    t = d.max(1.5 + rank)            # rank 1 is the slow one
    tokens_per_rank = 16384
    value = tokens_per_rank * d.world / (t / 1e3)
    out[rank] = (t, value, d.rank, d.world)
    d.close()


def test_two_rank_max_and_aggregate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5                       # max over ranks
    assert res[0][1] == pytest.approx(2 * 16384 / 2.5e-3)      # summed tokens / slowest time
    assert {res[0][2], res[1][2]} == {0, 1} and res[0][3] == 2


def _bench_cmd(*extra):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return [sys.executable, os.path.join(root, "bench.py"), *extra], root


def test_bench_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` with no launcher around it starts two ranks itself (torch.distributed.run
    on 127.0.0.1); the launcher check runs the barrier and the max over ranks on CPU (gloo) and
    reports the world size it saw."""
    import json
    import subprocess
    cmd, root = _bench_cmd("--gpus", "2", "--launcher-check")
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=240, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout        # rank 0 alone prints
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["launcher_check"] is True
    assert rec["max_rank_seconds"] >= 0.002  # the slower rank's time


def test_bench_refuses_disagreeing_world_size():
    import subprocess
    cmd, root = _bench_cmd("--gpus", "2", "--launcher-check")
    env = dict(os.environ, WORLD_SIZE="3", RANK="0", LOCAL_RANK="0")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120, env=env, cwd=root)
    assert r.returncode != 0 and "disagree" in r.stderr


def test_bench_reference_arm_prints_one_line():
    """`bench.py --impl reference` times the oracle on the host cores (no GPU) and prints one JSON
    line with the GPU arm's metric, the sample it ran, and an e2e entry with no copies."""
    import json
    import subprocess
    cmd, root = _bench_cmd("--impl", "reference", "--steps", "1", "--warmup", "1")
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    import bench
    assert rec["impl"] == "reference" and rec["metric"] == bench.METRIC and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["dtype"] == "f64"
    assert rec["steps"] == 1 and rec["warmup"] >= 1


def test_bench_reference_arm_other_ranks_exit_without_work():
    """Under a launcher with N > 1 only rank 0 runs the oracle arm; another rank exits 0 at once
    and prints nothing."""
    import subprocess
    import time
    cmd, root = _bench_cmd("--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1")
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    t = time.time()
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert time.time() - t < 120
