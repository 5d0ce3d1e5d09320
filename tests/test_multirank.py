"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2).

Under torchrun each rank runs its own replica of the step (the path shards
into independent problems: no data-path collective). The only cross-rank
steps are the timing reduction -- the job's step time is the slowest
rank's -- and, for the reference arm, that only rank 0 runs and prints.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.5 + rank              # rank 1 is the slow one
        worst = bench.max_over_ranks(ms, "cpu")
        tdist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"worst": worst, "value": bench.job_throughput(world, worst)}, f)
    finally:
        tdist.destroy_process_group()


def test_step_time_is_the_slowest_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    sys.path.insert(0, ROOT)
    import bench
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert [r["worst"] for r in res] == [2.5, 2.5]
    # whole-job throughput: both ranks' work over the slowest rank's time
    assert res[0]["value"] == pytest.approx(2 * bench.OPS_STEP / 2.5e-3 / 1e12)


def test_reference_arm_prints_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
