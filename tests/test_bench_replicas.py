"""The bench's N > 1 host logic on CPU: replicas (one process per GPU) report
the whole-job value from the slowest rank's time, reduced with all_reduce(MAX)
over a real process group (gloo, world size 2)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 100.0 + 50.0 * rank  # rank 1 is the slowest
        slowest = bench.max_over_ranks(torch, dist, my_ms, torch.device("cpu"))
        value = bench.aggregate_gbs(world, 2_000_000_000, 10, slowest)
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(f"{slowest} {value}")
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        slowest, value = map(float, (tmp_path / f"r{r}").read_text().split())
        assert slowest == 150.0
        # 2 ranks x 2 GB x 10 steps in 0.150 s
        assert abs(value - 2 * 2.0 * 10 / 0.150) < 1e-6
