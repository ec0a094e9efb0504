"""The multi-process paths of bench.py on CPU (gloo, world size 2): the
max-over-ranks timing reduction and the whole-job throughput, and the
reference arm under torchrun, where rank 0 alone runs and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 10 + r ms: every rank must see the slowest, 10 + world - 1
        out[rank] = bench.max_over_ranks(torch, 10.0 + rank)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_max_worker, args=(world, free_port(), out), nprocs=world, join=True)
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_max_over_ranks_single_process_and_throughput():
    assert bench.max_over_ranks(torch, 3.5) == 3.5
    # two ranks each streaming 1 GB per step for 10 steps in 5 ms: 4000 GB/s for the job
    assert bench.job_throughput(2, 10**9, 10, 5.0) == pytest.approx(4000.0)


def test_reference_arm_under_torchrun_rank0_only():
    env = dict(os.environ, QX_REF_STEP_S="0.2", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line_has_the_contract_keys():
    """One process, CPU only: the reference arm prints one JSON line with the
    keys the driver reads."""
    env = dict(os.environ, QX_REF_STEP_S="0.2", OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in j, k
    assert j["metric"] == bench.METRIC and j["unit"] == "GB/s" and j["higher_is_better"] is True
    assert j["steps"] == 1 and j["warmup"] == 3 and j["n_gpus"] == 1
    assert j["cpu_baseline"]["cores"] >= 1 and j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"]["value"] == j["value"] and j["e2e"]["unit"] == j["unit"]
