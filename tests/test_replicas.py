"""Host logic of the N-GPU bench on CPU: ranks are independent replicas of
the layer ("replicas only": the capacity rule is defined per batch, so no
step exchanges data), and the job's figures come from the slowest rank.
World size 2 over gloo on 127.0.0.1; no GPU."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")  # rank 1 is the slower replica
        q.put((rank, ms, bench.job_throughput(16384, world, ms)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time_and_throughput_counts_all_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, v in out:
        assert ms == 15.0  # every rank reports the slowest rank's time
        assert v == pytest.approx(2 * 16384 / 15e-3)  # both ranks' tokens over that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(100, 1, 2.0) == pytest.approx(50000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank but 0 leaves the reference arm at once,
    printing nothing (the oracle runs once, on rank 0's host cores)."""
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.parametrize("name,mode", [("tiny_fp32", "whole"), ("small_prefill", "experts"), ("training", "train")])
def test_cpu_baseline_runs_the_cpp_oracle_on_one_core(monkeypatch, name, mode):
    """bench.cpu_baseline on each of its modes, on small stand-ins of the
    workloads (inputs drawn on the host): the single-threaded C++ oracle
    runs, on one core, and the result says what it timed."""
    sys.path.insert(0, ROOT)
    import bench
    import moe_synth as S
    small = dict(tiny_fp32=S.WORKLOADS["tiny_fp32"].replace(T=32),
                 small_prefill=S.WORKLOADS["small_prefill"].replace(T=128, d=64, h=96, E=4),
                 training=S.WORKLOADS["training"].replace(T=64, d=64, h=96, E=4))
    monkeypatch.setitem(S.WORKLOADS, name, small[name])
    r = bench.cpu_baseline(name, mode=mode, max_rows=3)
    assert r["value"] > 0 and r["cores"] == 1 and r["kind"] == "oracle"
    assert r["impl"] == "C++ fp64 oracle, single thread"
    assert r["extrapolated"] == (mode != "whole")
    assert ("forward and backward" in r["sample"]) == (mode == "train")
