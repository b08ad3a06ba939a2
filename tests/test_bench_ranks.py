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


def test_dense_cpu_sample_rows_keep_their_keys():
    """The CPU sample (the last r query rows of every sequence against all of its keys, bottom-right)
    gives its rows the same O and dQ as the full problem, and counts 10 d FLOPs per visible pair."""
    import numpy as np
    import oracle
    import synth
    p = synth.dense_problem("s", dtype=synth.F16, b=2, h=2, h_kv=1, d=8, s_q=40, s_kv=40, mask=1, seed=3)
    q, k, v, do = (p.f64(x) for x in ("q", "k", "v", "do"))
    o, lse = oracle.dense_fwd(q, k, v, p.cu_q, p.cu_kv, p.scale, p.mask)
    dq, _, _ = oracle.dense_bwd(q, k, v, o, do, lse, p.cu_q, p.cu_kv, p.scale, p.mask)
    idx, take = bench._last_rows(p.cu_q, 7)
    assert take.tolist() == [7, 7] and idx.tolist() == list(range(33, 40)) + list(range(73, 80))
    cu = np.cumsum(take)
    so, slse = oracle.dense_fwd(q[idx], k, v, cu, p.cu_kv, p.scale, oracle.CAUSAL_BOTTOM_RIGHT)
    np.testing.assert_allclose(so, o[idx], rtol=1e-12, atol=1e-14)
    sdq, _, _ = oracle.dense_bwd(q[idx], k, v, so, do[idx], slse, cu, p.cu_kv, p.scale, oracle.CAUSAL_BOTTOM_RIGHT)
    np.testing.assert_allclose(sdq, dq[idx], rtol=1e-11, atol=1e-13)
    _, flops, _, units = bench.oracle_dense_sample(p, 7)
    pairs = 2 * sum(i + 1 for i in range(33, 40))  # top-left causal, equal lengths: row i sees keys 0 .. i
    assert flops == 10.0 * p.h * pairs * p.d and units == 2


def test_cpu_sample_sizes():
    """A full non-causal sample has the workload's FLOPs; units are (sequence, kv head) pairs."""
    import synth
    p = synth.workload(0)
    _, flops, _, units = bench.oracle_dense_sample(p)
    assert flops == bench.workload_info(0)[1] and units == p.b * p.h_kv
    q = synth.nsa_problem("n", dtype=synth.BF16, lens_q=[100, 50], lens_kv=[256, 256], n1=4, n2=2, d=128,
                          block_size=64, block_count=2, sparse_mode=2, seed=5)
    _, flops, _, units = bench.oracle_nsa_sample(q, 30)
    assert flops == 10.0 * 60 * 4 * 2 * 64 * 128 and units == 4


def _shard_rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = bench.shard_units(4, 12, rank)  # workload 1's shard: 4 sequences, 12 kv heads per rank
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        out[rank] = gathered
    finally:
        dist.destroy_process_group()


def test_shards_cover_every_unit_once_over_two_gloo_ranks():
    """Two gloo ranks: the union of their (sequence, kv head) units is the global problem's, with no
    unit on two ranks (so no collective is needed: every unit owns its dQ / dK / dV rows)."""
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_shard_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        units = [u for shard in out[rank] for u in shard]
        assert len(units) == len(set(units)) == world * 4 * 12
        assert set(units) == {(s, g) for s in range(world * 4) for g in range(12)}


def test_rank0_shard_is_the_workload():
    """Rank 0 of a sharded run holds exactly the single-GPU workload; other ranks hold the same shapes
    with their own draws."""
    import numpy as np
    import synth
    for idx in (1,):
        w, s0, s1 = synth.workload(idx), bench.shard_workload(idx, 0), bench.shard_workload(idx, 1)
        np.testing.assert_array_equal(w.q, s0.q)
        assert s1.q.shape[1:] == w.q.shape[1:] and not np.array_equal(s1.q[:10], w.q[:10])
        _, f0, _ = bench.workload_info(idx, s0)
        _, fw, _ = bench.workload_info(idx)
        assert f0 == fw
