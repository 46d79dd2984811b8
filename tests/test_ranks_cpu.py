"""The bench's N > 1 path on the CPU: two gloo ranks in separate processes
(the product does not shard, so each rank times its own replica; the only
exchanges are the timing barrier and the max over ranks of the step time)."""

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
    import time

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    try:
        # Rank 1 is slower: the barrier holds rank 0 until both have arrived.
        t0 = time.perf_counter()
        if rank == 1:
            time.sleep(0.3)
        dist.barrier()
        waited = time.perf_counter() - t0
        ms = 2.0 + rank                       # this rank's mean step time
        ms_max = bench.max_over_ranks(ms, dist, "cpu")
        value = bench.job_gflops(world, 5.0e10, ms_max)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{waited} {ms_max} {value}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_barrier(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    rows = {}
    for r in (0, 1):
        waited, ms_max, value = map(float, (tmp_path / f"rank{r}.txt").read_text().split())
        rows[r] = (waited, ms_max, value)
    # Both ranks see the slowest rank's time, and the job's rate counts both replicas.
    assert rows[0][1] == rows[1][1] == 3.0
    assert rows[0][2] == rows[1][2] == pytest.approx(2 * 5.0e10 / 3.0e-3 / 1e9)
    # Rank 0 waited at the barrier for the slower rank.
    assert rows[0][0] >= 0.25


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_gflops(1, 5.0e10, 1.25) == pytest.approx(5.0e10 / 1.25e-3 / 1e9)
