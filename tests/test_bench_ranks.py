"""bench.py's multi-replica host logic, on CPU with two gloo ranks.

With N GPUs the hot path runs as N independent replicas, one process per GPU
and no collective on the data path; the only cross-rank steps are the
barrier around the timed region and the maximum over ranks of the elapsed
time, and rank 0 alone prints.  The reference arm under torchrun runs on
rank 0 only; the other ranks exit at once without output."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if ROOT not in sys.path:
            sys.path.insert(0, ROOT)
        import bench
        # every rank times its own replica; the job's time is the slowest one
        mine = 0.25 + 0.5 * rank
        t = bench.max_over_ranks(mine, world, torch.device("cpu"))
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": t, "value": bench.job_throughput(1_000_000, 10, t, world)}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    slowest = 0.25 + 0.5 * (world - 1)
    for g in got:
        assert g["max"] == slowest
        # both replicas' bytes over the slowest rank's time
        assert g["value"] == pytest.approx(world * 1_000_000 * 10 / slowest / 1e9)


def test_job_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1, None) == 1.5
    assert bench.job_throughput(2_000_000_000, 3, 2.0, 1) == pytest.approx(3.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
