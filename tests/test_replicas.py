"""The multi-GPU path of the benchmark (independent replicas) with world_size 2 on CPU.

The block has no exchange step, so N GPUs run N replicas: the process group only
provides the barrier around the timed region and the max-over-ranks time. These
tests run that host logic under gloo, and the reference arm under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup("gloo")
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + r, w, device="cpu")  # rank 1 is the slower one
    v = bench.whole_job_gbs(3_000_000_000, t, w)
    q.put((r, w, t, v))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_replicas_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    for r, w, t, v in got:
        assert w == 2
        assert t == 2.0  # both ranks see the slowest rank's time
        assert abs(v - 2 * 3.0 / 2.0) < 1e-9  # 2 replicas x 3 GB over 2 s = 3 GB/s


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "tiny",
           "--ref-step-seconds", "0.05"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
