"""Multi-rank aggregation of the benchmark, on CPU with the gloo backend.

Sequences are independent, so N GPUs run N replicas with no collective on
the data path; the only cross-rank steps are the timing ones: the slowest
rank's time (max over ranks) and the whole-job throughput (all ranks' frames
over that time).  Two CPU ranks exercise exactly those helpers of bench.py.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out_dir: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [0.25, 0.75]                     # seconds each replica took
    slowest = bench.max_over_ranks(times[rank], "cpu")
    frames_per_rank = 256
    value = bench.replica_throughput(frames_per_rank, world, slowest)
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{slowest} {value}\n")
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_time_and_the_job_throughput(tmp_path):
    port = _free_port()
    mp.spawn(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        slowest, value = map(float, open(tmp_path / f"rank{r}.txt").read().split())
        assert slowest == 0.75                   # every rank sees the max
        assert value == pytest.approx(2 * 256 / 0.75)


def test_single_rank_throughput_is_plain():
    import bench
    assert bench.replica_throughput(240, 1, 2.0) == 120.0
