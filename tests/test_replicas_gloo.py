"""The bench's N-GPU form, replicas, exercised with two gloo processes on the
CPU: the barrier, the max over ranks of each time, the whole-job value, and
the reference arm's rule that only rank 0 works under torchrun."""
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch

    import bench

    r, lr, w = bench.dist_env()
    reps = bench.Replicas(w, "gloo", torch.device("cpu"))
    t0 = time.perf_counter()
    time.sleep(0.05 * (rank + 1))  # ranks finish at different times
    reps.barrier()
    mine = (time.perf_counter() - t0) * 1e3
    slowest = reps.reduce_max(mine)
    rate = reps.whole_job_rate(1000.0, slowest / 1e3)
    reps.close()
    q.put((r, lr, w, mine, slowest, rate))


def test_replicas_max_over_ranks_and_whole_job_value():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, lr0, w0, t0, s0, v0), (r1, lr1, w1, t1, s1, v1) = res
    assert (r0, r1, lr0, lr1, w0, w1) == (0, 1, 0, 1, 2, 2)
    assert s0 == s1 == max(t0, t1), "every rank reports the slowest rank's time"
    assert v0 == v1 == pytest.approx(2 * 1000.0 / (s0 / 1e3)), "units of all ranks / slowest time"


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun the reference arm runs on rank 0 only: rank 1 returns 0
    at once and prints nothing."""
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1"], env=env, capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""
