"""The multi-replica path of bench.py on CPU: two gloo ranks (the GPU runs use
the same code over NCCL).  The whole-job time per step is the slowest rank's
time over the steps of all ranks, and a non-zero rank of the reference arm
exits without output."""

import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, steps, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dist.barrier()
        v = bench.job_us_per_step(times[rank], steps, world)
        with open(os.path.join(out, f"r{rank}"), "w") as f:
            f.write(repr(v))
    finally:
        dist.destroy_process_group()


def test_whole_job_time_is_max_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    times, steps, world = [12.5, 30.0], 10, 2
    mp.start_processes(_rank, args=(world, _free_port(), times, steps, str(tmp_path)),
                       nprocs=world, start_method="spawn", join=True)
    got = [float(open(tmp_path / f"r{r}").read()) for r in range(world)]
    want = max(times) * 1e3 / (steps * world)
    assert got == [want, want]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_us_per_step(4.0, 8, 1) == 4.0 * 1e3 / 8


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
