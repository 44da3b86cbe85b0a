"""The N > 1 host path of bench.py with two gloo ranks on the CPU.

The path shards by batch rows with no exchange step, so N GPUs run N
independent replicas; the only collectives are the timing barrier and the
max-over-ranks reduction of the elapsed time. Here two ranks with different
local times must agree on the slowest one and on the whole-job rate.
"""
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms_local = 10.0 + 5.0 * rank              # rank 1 is the slower one
    dist.barrier()
    ms_max, rate = bench.replica_rate(ms_local, 1000.0, world, "cpu")
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms_max": ms_max, "rate": rate}, f)
    dist.destroy_process_group()


def test_two_replicas_agree_on_slowest_time_and_job_rate(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms_max"] == 15.0                        # the slower rank's time
        assert r["rate"] == pytest.approx(2 * 1000.0 / 0.015)   # both replicas' units over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms_max, rate = bench.replica_rate(4.0, 500.0, 1, "cpu")
    assert ms_max == 4.0 and rate == pytest.approx(500.0 / 0.004)
