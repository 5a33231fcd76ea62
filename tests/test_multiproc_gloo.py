"""The multi-rank path of bench.py on CPU: two ranks over the gloo backend
(rendezvous on 127.0.0.1) agree on the slowest rank's time, hold disjoint
agent blocks that cover the job, and report the whole-job throughput."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [40.0, 55.5][rank]                      # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        agents = list(bench.rank_agents(8, world, rank))
        everyone = [None] * world
        dist.all_gather_object(everyone, agents)
        out[rank] = (ms, agents, everyone, bench.job_tokens_per_s(8, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        ms, agents, everyone, value = res[rank]
        assert ms == 55.5                                  # the max over ranks, on every rank
        assert value == pytest.approx(2 * 8 / 55.5e-3)
    blocks = res[0][2]
    assert sorted(a for blk in blocks for a in blk) == list(range(16))   # disjoint, covering


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert list(bench.rank_agents(8, 1, 0)) == list(range(8))
    with pytest.raises(ValueError):
        bench.rank_agents(8, 2, 2)
