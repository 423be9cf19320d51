"""CPU checks of bench.py's multi-rank logic with world size 2 over gloo (127.0.0.1): the job time is the
max over ranks (the only collective), the whole-job value counts every replica's steps, and only rank 0
runs and prints the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local = [120.0, 150.0][rank]                       # this rank's timed region, ms
    job = bench.job_time_ms(local, world, "cpu")
    value = bench.whole_job_us_per_step(job, 50, world)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"job": job, "value": value}, f)


def test_job_time_is_max_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["job"] == 150.0                      # every rank sees the slowest replica
        assert d["value"] == pytest.approx(150.0 * 1e3 / (50 * 2))


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(12.5, 1) == 12.5
    assert bench.whole_job_us_per_step(12.5, 10, 1) == pytest.approx(1250.0)


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run_reference(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference(0, 2)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["higher_is_better"] is False and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["cores"] == (os.cpu_count() or 1)       # the oracle on every host core
