"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each reporting its own step
time, must both see the slowest one (the job's time is the maximum over ranks)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}"), "w") as f:
        f.write(repr(got))


@pytest.mark.timeout(120)
def test_two_ranks_agree_on_the_slowest_time(tmp_path):
    if not dist.is_available():
        pytest.skip("torch.distributed is not available")
    world = 2
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [float((tmp_path / f"rank{r}").read_text()) for r in range(world)]
    assert got == [2.5, 2.5]


def test_one_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.max_over_ranks(3.25, dist, "cpu") == 3.25  # no process group initialised
