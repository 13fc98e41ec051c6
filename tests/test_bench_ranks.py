"""bench.py's multi-rank timing on the CPU: two gloo ranks, each a replica
with its own step time; the reported time is the slowest rank's and the
value counts the tokens of every rank."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [0.004 + 0.002 * rank, 1.0 + rank, 3.0 - rank]
    got = bench.reduce_max_over_ranks(mine)
    out.put((rank, got, bench.whole_job_tokens_per_s(world, 4096, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [0.006, 2.0, 3.0]
        assert abs(value - 2 * 4096 / 0.006) < 1e-6


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([1.0, 2.0]) == [1.0, 2.0]
    assert bench.whole_job_tokens_per_s(1, 4096, 0.004) == 4096 / 0.004
