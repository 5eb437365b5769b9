"""The N > 1 launch path on CPU: world-size-2 process groups on gloo.

The path shards by tokens with no exchange (replicas only), so the only
cross-rank logic is the timing reduction (maximum over ranks) and the
reference arm, which rank 0 alone runs and prints. Both are exercised here
with two gloo ranks, no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports times (r + 1, 10 - r): the maximum over ranks is (world, 10)
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], torch.device("cpu"))
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_the_maximum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got[0] == got[1] == [2.0, 10.0]


def test_max_over_ranks_without_a_process_group_is_the_identity():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.0], torch.device("cpu")) == [3.5, 1.0]


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny",
           "--cpu-sample-tokens", "4"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
