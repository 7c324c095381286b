"""bench.py's multi-process logic on CPU: two gloo ranks (world size 2)
exercise the barrier and the max / sum reductions the benchmark uses to turn
per-rank replica timings into one whole-job number, and the reference arm's
rule that only rank 0 times and prints."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    ms = 10.0 + 5.0 * r                       # rank 1 is the slow one
    out[r] = (bench.max_over_ranks(ms, w), bench.sum_over_ranks(1.0, w))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    world, port = 2, free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == (15.0, 2.0)


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_reference_arm_relaunches_itself_with_two_ranks():
    """--gpus 2 without a launcher: bench.py starts torch.distributed.run with
    two ranks; rank 0 alone times the oracle and prints one line."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["MASTER_PORT"] = str(free_port())
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    import json
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
