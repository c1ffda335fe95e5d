"""The benchmark's multi-rank bookkeeping with a world-size-2 gloo group on
CPU: every rank owns a disjoint shard of heads of a job twice as large (weak
scaling, no data crosses ranks), the step time is the maximum over ranks and
the whole-job value counts the work of every shard."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    got = bench.max_over_ranks(ms, "cpu")
    heads = bench.shard_heads(rank, world, 24)
    # every rank learns every shard (a test-only gather; the benchmark exchanges nothing)
    shards = [None] * world
    dist.all_gather_object(shards, heads)
    out[rank] = (got, bench.whole_job_tflops(2e12, world, got), shards)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == 5.0 and out[1][0] == 5.0
    # two replicas of 2e12 flops in 5 ms: 800 TFLOP/s for the whole job
    assert out[0][1] == pytest.approx(800.0)
    shards = out[0][2]
    assert shards == out[1][2]
    assert sorted(shards[0] + shards[1]) == list(range(48))          # disjoint, cover the job
    assert len(shards[0]) == len(shards[1]) == 24                      # fixed work per rank


def test_shard_heads_rejects_bad_ranks():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(ValueError):
        bench.shard_heads(2, 2, 24)
    with pytest.raises(ValueError):
        bench.shard_heads(0, 1, 0)
