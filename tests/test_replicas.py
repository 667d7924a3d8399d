"""Multi-GPU here means independent replicas (decode attention shards by
sequence with no exchange). The host logic -- per-rank replica batches, the
max-over-ranks time and the whole-job rate -- runs as two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [10.0, 25.0][rank]
        worst = bench.max_over_ranks(my_ms, world)
        rate = bench.whole_job_rate(64, 100, world, worst)
        from paged_kv_decode_18_gb300 import workloads as W
        w = W.tiny(seed=bench.replica_seed(1, rank), num_seqs=2, lo=20, hi=40, num_blocks=8)
        sig = int(w.q.view(torch.int16).to(torch.int64).sum())
        q.put((rank, worst, rate, sig))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, w0, r0, s0), (_, w1, r1, s1) = res
    assert w0 == w1 == 25.0                       # both ranks see the slowest time
    assert r0 == r1 == pytest.approx(2 * 64 * 100 / 0.025)
    assert s0 != s1                               # each rank has its own replica batch


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(64, 10, 1, 1000.0) == pytest.approx(640.0)
