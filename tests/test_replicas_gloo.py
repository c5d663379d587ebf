"""The multi-GPU path of the benchmark is replicas only (the step needs no
exchange between GPUs): each rank runs its own step and the job reports the
slowest rank's time.  Checked here with two gloo ranks on the CPU."""
import json
import os
import socket
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
    mine = [0.25 + 0.5 * rank, 1.0 + rank]     # ms per step, e2e seconds: rank 1 is slower
    got = bench.reduce_max(mine, world)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"got": got, "value": bench.job_tokens_per_s(512, world, got[0] / 1e3)}, f)


def test_two_replicas_report_the_slowest_rank(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["got"] == [0.75, 2.0]
        assert abs(d["value"] - 2 * 512 / 0.75e-3) < 1e-6


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([3.0, 4.0], 1) == [3.0, 4.0]
