"""The multi-GPU path of bench.py runs independent replicas, one per rank, and
reports the whole job's throughput over the slowest rank's time.  Its rank
arithmetic runs here on CPU with two gloo ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
        out[rank] = bench.slowest_rank_ms(local_ms, dist, "cpu")
    finally:
        dist.destroy_process_group()


def test_slowest_rank_over_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 20.0


def test_single_rank_and_job_throughput():
    assert bench.slowest_rank_ms(7.5) == 7.5
    flops = 1.0e12  # per replica and step
    # two replicas, 2 ms per step on the slowest: 2 * 1e12 / 2e-3 s = 1000 TFLOP/s
    assert bench.job_tflops(2, flops, 2.0) == pytest.approx(1000.0)
    assert bench.job_tflops(1, flops, 2.0) == pytest.approx(500.0)


def test_time_repeated_reaches_the_minimum():
    """The CPU-baseline timer repeats a short sample until the minimum time has passed."""
    import time
    import bench
    calls = []
    n, dt = bench.time_repeated(lambda: (calls.append(1), time.sleep(0.01)), 0.05)
    assert n == len(calls) and n >= 5 and dt >= 0.05
    n, dt = bench.time_repeated(lambda: time.sleep(0.02), 0.0)
    assert n == 1  # always at least once


def test_sample_threads_counts_what_the_oracle_uses():
    """The oracle runs one thread per (sequence, kv head) unit at most; a CPU sample covers one sequence."""
    import oracle
    import synth
    assert bench.sample_threads(synth.workload(1)) == min(oracle.thread_count(), 12)
    assert bench.sample_threads(synth.workload(4)) == 1
