"""The N > 1 path of bench.py without a GPU: replicas only (no collective on
the data path), so the host logic is the slowest-replica time and the
whole-job throughput, plus rank 0 alone printing. Checked with two gloo ranks
on the CPU, and by running the reference arm under torchrun with two ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
        q.put((rank, slowest, bench.job_throughput(world, 2e12, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, tput in got:
        assert slowest == 15.0
        assert tput == pytest.approx(2 * 2e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(key, None)
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_throughput(1, 1e12, 1.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-rows", "2",
           "--workload", "gqa4_s256_d128_fp16"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
