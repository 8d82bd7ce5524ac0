"""The multi-process (replica) aggregation of bench.py, on CPU with the gloo backend.

The hot path shards by request, so N GPUs run N independent replicas with no
collective on the data path; the only cross-rank step is the timing: the job
is as slow as its slowest rank, and its throughput counts every rank's tokens.
Two gloo ranks with different local times must both see the maximum, and the
reported throughput must be world * units / max time.
"""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], "cpu")
        value = bench.replica_throughput(64, world, ms)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {value!r}\n")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_timing_is_max_over_ranks(tmp_path, world):
    import torch.multiprocessing as mp
    times = [0.25, 0.5]
    mp.spawn(_rank_main, args=(world, _free_port(), times, str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        ms, value = map(float, open(tmp_path / f"r{r}.txt").read().split())
        assert ms == max(times)
        assert value == pytest.approx(64 * world / (max(times) / 1000.0))


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.replica_throughput(64, 1, 0.5) == pytest.approx(128000.0)
