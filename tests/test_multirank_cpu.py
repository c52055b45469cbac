"""The N > 1 path of bench.py on CPU: two gloo ranks, as torchrun would start
them.  Each rank runs an independent replica (weak scaling), the job's time
is the slowest rank's, and the whole-job rate counts every rank's work; the
reference arm runs on rank 0 only and the other ranks exit 0 silently."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # each rank reports a different elapsed time; all must agree on the max
        elapsed = 10.0 + 5.0 * rank
        bench.barrier(world)
        m = bench.max_over_ranks(elapsed, world)
        q.put((rank, m, bench.job_rate(2e12, 100, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[1] for g in got] == [15.0, 15.0]
    # 2 ranks x 100 steps x 2 TFLOP in 15 ms
    assert all(abs(g[2] - 2e12 * 2 * 100 / 15e-3 / 1e12) < 1e-6 for g in got)


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "worked_9x9", "--steps", "1", "--warmup", "0"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "worked_9x9", "--steps", "2", "--warmup", "1"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0
    import json
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
