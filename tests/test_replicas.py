"""The N > 1 path on CPU: two gloo ranks aggregate timings the way bench.py does
(slowest rank, whole-job throughput), with distinct per-rank seeds."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from skinny_bf16_gemm_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, l = replicas.rank_info()
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        slow = replicas.slowest_ms(ms)
        gbs = replicas.aggregate_throughput(1_000_000_000, 4, slow, w)
        out[rank] = (r, w, l, slow, gbs, replicas.replica_seed(123, r))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, l, slow, gbs, seed) in res.items():
        assert (r, w, l) == (rank, world, rank)
        assert slow == pytest.approx(15.0)
        assert gbs == pytest.approx(2 * 1e9 * 4 / 15e-3 / 1e9)
    assert res[0][5] != res[1][5]


def test_single_process_is_its_own_slowest():
    assert replicas.slowest_ms(3.5) == 3.5
    assert replicas.aggregate_throughput(2_000_000_000, 2, 1.0, 1) == pytest.approx(4000.0)
