"""The multi-GPU path of the benchmark, exercised on CPU with two gloo ranks.

The product shards with no data exchange (output tiles are independent), so
N GPUs run N replicas; the only cross-rank steps are the barrier around the
timed region and the max over ranks of the timed seconds, from which the
whole-job throughput is computed.  Both run here as two processes over gloo
on 127.0.0.1; the reference arm's rank rule (rank 0 alone works and prints)
runs as two plain processes.
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        tdist.barrier()
        # each rank "timed" a different total; the job takes the slowest
        mine = [0.25, 0.4][rank]
        slowest = bench.max_over_ranks(mine, ws)
        value = bench.job_throughput(ws, 10, 2.0e9, slowest)
        out.put((rank, slowest, value))
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank_and_the_job_throughput():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, slowest, value in got:
        assert slowest == 0.4
        # 2 ranks x 10 steps x 2 GFLOP over 0.4 s
        assert value == pytest.approx(2 * 10 * 2.0 / 0.4)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(1, 4, 1e9, 2.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only():
    base = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", LOCAL_RANK="0")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "s1_128", "--steps", "1", "--warmup", "3"]
    r1 = subprocess.run(cmd, env=dict(base, RANK="1"), capture_output=True, text=True,
                        timeout=120)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(cmd, env=dict(base, RANK="0"), capture_output=True, text=True,
                        timeout=300)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_timing_rule_follows_the_operand_size():
    # Workloads whose operands are larger than L2 (129 MB) run back to back
    # without a flush; the others are flushed before every step.  The rule
    # and the config note the line carries agree, and both arms share them.
    streamed = {n for n in bench.WORKLOADS if bench.streams_past_l2(bench.datagen.CONFIGS[n])}
    assert {"s3_4092", "s4_rect", "s6_skinny", "s7_gemv", "s9_ax"} <= streamed
    assert not streamed & {"s1_128", "s2_2048", "s5_odd", "s8_2049"}
    for n in bench.WORKLOADS:
        cfg = bench.datagen.CONFIGS[n]
        big = bench.algorithmic_bytes(cfg) > bench.L2_BYTES_GB300
        assert (n in streamed) == big
        note = bench.workload_config(n)["l2"]
        assert ("back to back" in note) == big and ("flushed before every timed step" in note) != big
