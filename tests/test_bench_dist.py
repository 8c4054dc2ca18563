"""Host logic of the multi-GPU benchmark path (replicas, no collective on the
data path), run as world-size-2 process groups on the gloo backend on CPU."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out_path):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r processed 1000 * (r + 1) units in 10 * (r + 1) ms
        value, ms = bench.job_throughput(1000.0 * (rank + 1), 10.0 * (rank + 1), world)
        if rank == 0:
            with open(out_path, "w") as f:
                json.dump({"value": value, "ms": ms}, f)
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_job_throughput_sums_units_and_takes_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    out = str(tmp_path / "r0.json")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    d = json.load(open(out))
    assert d["ms"] == 20.0
    assert abs(d["value"] - 3000.0 / 0.020) < 1e-6


def test_job_throughput_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    v, ms = bench.job_throughput(500.0, 250.0, 1)
    assert ms == 250.0 and abs(v - 2000.0) < 1e-9


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--ref-frames", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line(orc):
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--ref-frames", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "codes/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
