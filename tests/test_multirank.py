"""Host side of the multi-rank bench path on CPU (gloo, world_size 2): each
rank works on its own shard of heads with no collective on the data path, and
the reported time is the maximum over ranks, reached through a barrier."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    assert (d.rank, d.world) == (rank, world)
    d.init("gloo")
    d.barrier()
    # a slower rank decides the reported time
    t = d.max(1.5 if rank == 1 else 0.25)
    seed = bench.shard_seed(1003, rank)
    d.barrier()
    d.done()
    out.put((rank, t, seed))


def test_two_ranks_report_the_slowest_and_draw_distinct_shards():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], f"rank exit codes {codes}"
    res = sorted(out.get() for _ in range(world))
    assert [r[1] for r in res] == [1.5, 1.5]
    assert res[0][2] != res[1][2]


def test_single_rank_needs_no_process_group(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    d = bench.Dist()
    d.init("nccl")       # world 1: no process group is created
    assert d.pg is None and d.max(3.0) == 3.0
    d.barrier()
    d.done()
