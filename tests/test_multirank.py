"""The multi-GPU path of the benchmark on CPU: N independent replicas, no
collective on the data path, the job's step time is the slowest rank's and
its throughput the sum over ranks (world_size-2 gloo process group)."""

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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [3.0, 5.0][rank]
        mean = bench.job_mean_ms(local, world, torch.device("cpu"))
        out[rank] = (mean, bench.job_tflops(1e12, mean, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_throughput_sums_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        mean, tflops = res[r]
        assert mean == 5.0
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.job_mean_ms(4.0, 1, None) == 4.0
    assert bench.job_tflops(2e12, 4.0, 1) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_sweep_resumes_after_recorded_workloads(tmp_path):
    path = tmp_path / "sweep.jsonl"
    h = bench.kernel_hash()
    lines = [
        {"config": {"workload": "a"}, "kernel_hash": h},
        {"config": {"workload": "b"}, "kernel_hash": "other"},   # older kernel: redo
        "not json",
        {"config": {"workload": "c"}, "kernel_hash": h},
    ]
    with open(path, "w") as f:
        for x in lines:
            f.write((x if isinstance(x, str) else __import__("json").dumps(x)) + "\n")
    assert bench.sweep_todo(str(path), ["a", "b", "c", "d"], h) == ["b", "d"]
    assert bench.sweep_todo(str(tmp_path / "missing.jsonl"), ["a", "b"], h) == ["a", "b"]
