"""Multi-rank host logic of the benchmark on CPU (gloo, world_size 2).

The LiSA layer needs no collective on its data path: every rank runs its own
batch of (batch, head) slices.  What the ranks share is the timing: the job
time is the slowest rank's, and the reported value is all ranks' units over
that time.  The reference arm runs on rank 0 only and prints one line."""
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

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
    ms_max = bench.max_over_ranks(local_ms, world)
    value = bench.weak_throughput(world, 100352, 7, ms_max)
    out[rank] = (ms_max, value)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_throughput_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        ms_max, value = out[rank]
        assert ms_max == 15.0
        assert value == pytest.approx(2 * 100352 * 7 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_throughput(1, 10, 4, 2.0) == pytest.approx(20000.0)


def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` launched as two ranks: rank 0 times the
    oracle and prints exactly one JSON line, rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "deit_t_14x14"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["unit"] == bench.UNIT and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_metric_strings_format():
    """Both metric strings of the JSON line format without error (a literal
    percent sign in a format string once broke the backward line)."""
    assert "%" not in bench.METRIC.replace("% of", "")
    for extra in ("", " and the MLP parameters"):
        line = bench.BWD_METRIC % extra
        assert line.endswith("% of HBM roofline") and extra in line


def test_roofline_bytes_scale_with_width_and_dtype():
    """The per-kernel byte table is per token*head at bf16, d = 64; narrower
    widths and fp32 scale it, never to zero."""
    assert bench.stage_bytes("epilogue", 196, 16, "f32") == 196 * 4 * 16 * 4      # Q, K, V, O in fp32
    assert bench.stage_bytes("tc_epilogue", 100352, 64, "bf16") == 100352 * 512
    assert bench.stage_bytes("tc_stats_fused", 10, 64, "bf16") == 10 * 384
    assert bench.stage_bytes("tc_recur", 10, 64, "bf16") == 0
