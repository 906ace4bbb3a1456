"""The N > 1 path of bench.py on the CPU: ranks as processes over the gloo backend.

The layer has no exchange step (replicas only), so what is shared across ranks is host logic:
the slowest rank's time, the whole-job rate, and the reference arm, which rank 0 alone runs and
prints under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        max_ms = bench.max_over_ranks(local_ms, dist, device="cpu")
        results.put((rank, max_ms, bench.whole_job_rate(4096, 100, world, max_ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(results.get(timeout=10) for _ in range(world))
    for rank, max_ms, rate in got:
        assert max_ms == 15.0                            # every rank sees the slowest rank's time
        assert rate == pytest.approx(4096 * 100 * 2 / 0.015)


def test_whole_job_rate_single_rank():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_rate(32, 10, 1, 2.0) == pytest.approx(160000.0)


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, PYTHONPATH=ROOT, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "tiny_f32", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                               # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
