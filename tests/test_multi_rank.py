"""bench.py's N > 1 path on CPU, with two gloo ranks.

The verify step of one sequence has no exchange step, so N > 1 runs one
independent replica per rank. What the job adds is host logic: the timed
region is the slowest rank's, the whole-job value counts every replica's
steps, and the reference arm runs on rank 0 alone, the other ranks exiting
without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = 100.0 + 25.0 * rank                 # rank 1 is the slower replica
    m = bench.max_over_ranks(ms, world, "cpu")
    q.put((rank, m, bench.job_steps_per_s(m, 10, world)))
    tdist.destroy_process_group()


def test_two_ranks_time_the_slowest_replica_and_count_every_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [125.0, 125.0]
    # 10 steps on each of 2 replicas within the slowest rank's 125 ms
    assert out[0][2] == pytest.approx(160.0)
    assert out[1][2] == pytest.approx(160.0)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(42.5, 1, "cpu") == 42.5
    assert bench.job_steps_per_s(500.0, 100, 1) == pytest.approx(200.0)


def test_reference_arm_under_torchrun_prints_on_rank_zero_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle"
