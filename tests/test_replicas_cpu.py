"""The multi-GPU path of bench.py is replicas only (each rank runs the same
workload on its own GPU, no collective on the data path); its host logic is
checked here on CPU with the gloo backend and world size 2: the slowest
rank's time is taken over ranks and the whole-job value counts the units of
all ranks over that time; under torchrun the reference arm runs on rank 0
only and prints one line."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_rank = [2.0, 3.0][rank]           # rank 1 is the slower one
    value_rank = 100.0 / ms_rank         # units per ms on this rank (100 units each)
    ms = bench.max_over_ranks(ms_rank, dist, "cpu")
    out[rank] = (ms, bench.job_value(value_rank, ms_rank, ms, world))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    for r in range(2):
        ms, value = out[r]
        assert ms == 3.0                      # every rank sees the slowest time
        assert value == pytest.approx(200.0 / 3.0)  # 2 x 100 units over 3 ms


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
    assert bench.job_value(10.0, 1.0, 1.0, 1) == 10.0


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
